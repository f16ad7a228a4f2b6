"""CPU checks of the C ABI: the library builds, loads without a GPU, exports every
function `include/ridgefill.h` declares, and its host helpers and struct layouts
agree with the header."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ridgefill.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ridgefill_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    from late_layer_kv_gb300 import library_path
    out = subprocess.run(["nm", "-D", "--defined-only", library_path()], capture_output=True,
                         text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), f"{n} missing from the dynamic symbol table"


def test_compute_share_helper_matches_printed_ceilings(lib):
    from late_layer_kv_gb300 import compute_share
    for N, sp in ((9216, 1.64), (16384, 1.78), (32768, 1.88)):
        assert abs(1.0 / compute_share(24, 48, 2048, N) - sp) <= 0.005


def _c_sizeof(struct):
    code = f'#include "ridgefill.h"\n#include <stdio.h>\n#include <stddef.h>\nint main(void){{printf("%zu", sizeof({struct}));return 0;}}\n'
    exe = os.path.join(tempfile.mkdtemp(prefix="rf_sizeof_"), "sizeof_" + struct)
    r = subprocess.run(["gcc", "-x", "c", "-I", os.path.join(ROOT, "include"), "-o", exe, "-"],
                       input=code, text=True, capture_output=True)
    if r.returncode != 0:
        pytest.skip("no C compiler")
    return int(subprocess.run([exe], capture_output=True, text=True).stdout)


def _c_offsets(struct, fields):
    body = "".join(f'printf("%zu\\n", offsetof({struct}, {f}));' for f in fields)
    code = (f'#include "ridgefill.h"\n#include <stdio.h>\n#include <stddef.h>\n'
            f'int main(void){{{body}return 0;}}\n')
    exe = os.path.join(tempfile.mkdtemp(prefix="rf_offsetof_"), "offsetof_" + struct)
    r = subprocess.run(["gcc", "-x", "c", "-I", os.path.join(ROOT, "include"), "-o", exe, "-"],
                       input=code, text=True, capture_output=True)
    assert r.returncode == 0, r.stderr
    return [int(x) for x in subprocess.run([exe], capture_output=True, text=True).stdout.split()]


def test_ctypes_field_offsets_match_header():
    """Every field of the binding's structs sits at the header's offset, under the header's
    name."""
    from late_layer_kv_gb300 import ridgefill as rb
    for cls, struct in ((rb.FillArgs, "rf_fill_args"), (rb.GdnArgs, "rf_gdn_args"),
                        (rb.FitArgs, "rf_fit_args"), (rb.RescaleArgs, "rf_rescale_args"),
                        (rb.QuantizeArgs, "rf_quantize_args")):
        names = [f[0] for f in cls._fields_]
        header_names = {"lam": "lambda"}  # a Python keyword in the binding
        offs = _c_offsets(struct, [header_names.get(n, n) for n in names])
        assert offs == [getattr(cls, n).offset for n in names], struct


def test_abi_version_matches_binding(lib):
    from late_layer_kv_gb300 import ridgefill as rb
    assert lib.ridgefill_abi_version() == rb.ABI_VERSION


def test_ctypes_structs_match_header():
    from late_layer_kv_gb300 import ridgefill as rb
    assert ctypes.sizeof(rb.FillArgs) == _c_sizeof("rf_fill_args")
    assert ctypes.sizeof(rb.GdnArgs) == _c_sizeof("rf_gdn_args")
    assert ctypes.sizeof(rb.FitArgs) == _c_sizeof("rf_fit_args")
    assert ctypes.sizeof(rb.RescaleArgs) == _c_sizeof("rf_rescale_args")
    assert ctypes.sizeof(rb.QuantizeArgs) == _c_sizeof("rf_quantize_args")


def test_invalid_arguments_fail_without_a_gpu(lib):
    from late_layer_kv_gb300 import ridgefill as rb
    a = rb.FillArgs()
    a.n_layers = 1
    a.d_in = 100  # not a multiple of 64
    a.d_out = 256
    a.n_kv_heads = 2
    a.head_dim = 64
    assert lib.ridgefill_fill_workspace_size(ctypes.byref(a)) == 0
    assert lib.ridgefill_fill(ctypes.byref(a), None, 0, None) == 2  # RF_ERR_SHAPE
    assert b"d_in" in lib.ridgefill_last_error()
    assert lib.ridgefill_status_string(2) == b"unsupported or inconsistent shape"


def test_workspace_size_formula(lib):
    from late_layer_kv_gb300 import ridgefill as rb
    a = rb.FillArgs(20, 4096, 4096, 8, 128, 0, 14336, 0, 16384, 0, 5e5, 1e-6)
    ws = lib.ridgefill_fill_workspace_size(ctypes.byref(a))
    xhat = 20 * 14336 * 4096 * 2
    ss = 20 * (4096 // 256) * 14336 * 4
    rope = 64 * 14336 * 8  # (cos, sin) f32 pairs of the chunk's positions
    assert xhat + ss + rope <= ws <= xhat + ss + rope + 1024


def test_generic_workspace_size_matches_each_call(lib):
    """ridgefill_workspace_size(which, args) answers as the per-call size functions."""
    from late_layer_kv_gb300 import ridgefill as rb
    lib.ridgefill_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_void_p]
    lib.ridgefill_workspace_size.restype = ctypes.c_size_t
    fa = rb.FillArgs(20, 4096, 4096, 8, 128, 0, 14336, 0, 16384, 0, 5e5, 1e-6)
    ga = rb.GdnArgs()
    ga.n_layers, ga.d_in, ga.d_out, ga.n_heads, ga.d_k, ga.d_v, ga.chunk = 15, 4096, 4096, 16, 128, 128, 64
    ga.rows, ga.rms_eps, ga.l2_eps = 28672, 1e-6, 1e-6
    ta = rb.FitArgs()
    ta.n_layers, ta.d_in, ta.d_out, ta.flags, ta.rows, ta.lam = 20, 4096, 4096, 3, 65536, 1e-3
    ra = rb.RescaleArgs()
    ra.n_layers, ra.d_in, ra.d_out, ra.n_kv_heads, ra.head_dim, ra.which = 20, 4096, 4096, 8, 128, 1
    ra.tail_rows, ra.rows, ra.pos0, ra.cache_len, ra.rms_eps = 512, 14336, 0, 16384, 1e-6
    pairs = [(0, fa, lib.ridgefill_fill_workspace_size), (1, ga, lib.ridgefill_gdn_workspace_size),
             (2, ta, lib.ridgefill_fit_workspace_size), (3, ra, lib.ridgefill_rescale_workspace_size)]
    for which, args, single in pairs:
        ws = lib.ridgefill_workspace_size(which, ctypes.cast(ctypes.byref(args), ctypes.c_void_p))
        assert ws > 0 and ws == single(ctypes.byref(args))
    assert lib.ridgefill_workspace_size(7, ctypes.cast(ctypes.byref(fa), ctypes.c_void_p)) == 0
    assert b"unknown call" in lib.ridgefill_last_error()
    assert lib.ridgefill_workspace_size(0, None) == 0


def _fill_ok(rb):
    a = rb.FillArgs()
    a.n_layers, a.d_in, a.d_out, a.n_kv_heads, a.head_dim = 2, 256, 256, 2, 64
    a.rows, a.cache_len, a.rope_theta, a.rms_eps = 100, 128, 1e4, 1e-6
    return a


def test_new_argument_checks_fail_without_a_gpu(lib):
    """Argument errors of the exact-row, int8, host split-state, quantizer, rescale and
    GDN options are reported before anything is enqueued (no device needed)."""
    from late_layer_kv_gb300 import ridgefill as rb
    RF_ERR_ARG, RF_ERR_SHAPE = 1, 2
    a = _fill_ok(rb)
    assert lib.ridgefill_fill_workspace_size(ctypes.byref(a)) > 0
    idx = (ctypes.c_int32 * 4)(0, 1, 2, 3)
    a.row_idx = ctypes.cast(idx, ctypes.c_void_p)
    a.h_rows = 50  # fewer prefix rows than rows to fill
    assert lib.ridgefill_fill(ctypes.byref(a), None, 0, None) == RF_ERR_SHAPE
    a.h_rows, a.cache_len = 200, 128  # positions past the cache
    assert lib.ridgefill_fill(ctypes.byref(a), None, 0, None) == RF_ERR_SHAPE
    a.cache_len, a.h_on_host = 256, 1  # host split state with a row list
    assert lib.ridgefill_fill(ctypes.byref(a), None, 0, None) == RF_ERR_ARG
    a = _fill_ok(rb)
    a.h_on_host = 2
    assert lib.ridgefill_fill(ctypes.byref(a), None, 0, None) == RF_ERR_ARG
    a = _fill_ok(rb)
    a.d_in, a.A_scale = 192, 16  # int8 maps need d_in % 128 == 0
    assert lib.ridgefill_fill(ctypes.byref(a), None, 0, None) == RF_ERR_SHAPE

    q = rb.QuantizeArgs(1, 256, 192, 0, None, None, None)  # d_in not a multiple of 128
    assert lib.ridgefill_quantize_maps(ctypes.byref(q), None) == RF_ERR_SHAPE
    q = rb.QuantizeArgs(1, 256, 256, 0, None, None, None)
    assert lib.ridgefill_quantize_maps(ctypes.byref(q), None) == RF_ERR_ARG
    q = rb.QuantizeArgs(1, 256, 256, 3, 16, 16, 16)
    assert lib.ridgefill_quantize_maps(ctypes.byref(q), None) == RF_ERR_ARG

    r = rb.RescaleArgs()
    r.n_layers, r.d_in, r.d_out, r.n_kv_heads, r.head_dim = 2, 256, 256, 2, 64
    r.which, r.tail_rows, r.rows, r.cache_len, r.rms_eps = 3, 10, 0, 128, 1e-6
    assert lib.ridgefill_rescale(ctypes.byref(r), None, 0, None) == RF_ERR_ARG  # bad `which`
    r.which, r.tail_rows = 1, 0
    assert lib.ridgefill_rescale(ctypes.byref(r), None, 0, None) == RF_ERR_ARG  # no tail rows

    g = rb.GdnArgs()
    g.n_layers, g.d_in, g.d_out, g.n_heads, g.d_k, g.d_v, g.chunk = 1, 256, 256, 8, 128, 128, 64
    g.rows, g.rms_eps, g.l2_eps = 100, 1e-6, 1e-6
    g.S = 16
    g.n_exact = 101  # more exact rows than rows
    assert lib.ridgefill_fill_gdn(ctypes.byref(g), None, 0, None) == RF_ERR_ARG
    g.n_exact = 5  # exact rows without their indices and inputs
    assert lib.ridgefill_fill_gdn(ctypes.byref(g), None, 0, None) == RF_ERR_ARG


def test_map_source_arguments_fail_without_a_gpu(lib):
    """A host map source needs maps_on_host = 1 and a non-negative wait bound; both are
    checked before anything is enqueued."""
    from late_layer_kv_gb300 import ridgefill as rb
    a = _fill_ok(rb)
    a.map_source = rb.MAP_SOURCE_FN(lambda user, layer, dst, n: 0)
    assert lib.ridgefill_fill(ctypes.byref(a), None, 0, None) == 1  # maps_on_host = 0
    assert b"maps_on_host" in lib.ridgefill_last_error()
    a.maps_on_host, a.host_wait_ms = 1, -1
    assert lib.ridgefill_fill(ctypes.byref(a), None, 0, None) == 1
    assert lib.ridgefill_status_string(9) == b"the host map source reported an error"


def test_debug_library_builds_and_adds_guard_bands():
    """The debug build (RF_DEBUG=1) loads without a GPU, exports the same symbols, and its
    workspaces hold one guard band after every region: the fill of a resident-map call has
    seven regions (predicted inputs, partial sums, map slots, row gather, host split
    state, RoPE table, int8 layer groups), the fit with both steps thirteen (column-sum
    partials; G^, scales, two means, alpha, L^-1 copies, held-back panel blocks, inverse
    planes, G^-1, both solve operands, offset partials)."""
    from late_layer_kv_gb300 import build as b
    from late_layer_kv_gb300 import ridgefill as rb
    dbg = rb.load(debug=True)
    rel = rb.load(debug=False)
    for n in _declared():
        assert hasattr(dbg, n), f"{n} not exported by the debug library"
    assert dbg.ridgefill_abi_version() == rel.ridgefill_abi_version()
    fa = rb.FillArgs(20, 4096, 4096, 8, 128, 0, 14336, 0, 16384, 0, 5e5, 1e-6)
    ta = rb.FitArgs()
    ta.n_layers, ta.d_in, ta.d_out, ta.flags, ta.rows, ta.lam = 20, 4096, 4096, 3, 65536, 1e-3
    guard = 4096
    assert (dbg.ridgefill_fill_workspace_size(ctypes.byref(fa)) ==
            rel.ridgefill_fill_workspace_size(ctypes.byref(fa)) + 7 * guard)
    assert (dbg.ridgefill_fit_workspace_size(ctypes.byref(ta)) ==
            rel.ridgefill_fit_workspace_size(ctypes.byref(ta)) + 13 * guard)
    assert os.path.basename(b.LIB_DEBUG) == "libridgefill_debug.so"
