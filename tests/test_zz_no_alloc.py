"""ridgefill_fill_noalloc, the fill for callers that cannot allocate device memory.

Some callers (a host engine that owns every device buffer, or code running
after the engine has divided up all device memory) can pass inputs and
outputs but no workspace.  This entry point keeps its scratch in a
library-owned static device array.  Here it is called through the C ABI and
checked bit for bit against ridgefill_fill on two calls in a row: the second
call must not be affected by what the first left in the shared array.

This file is named to run last in a full test session; it also passes alone.
"""
import ctypes

import pytest
import torch

from synthetic import FillShape, fill_inputs
from tests._fill_helpers import SENTINEL, new_cache, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import device_error, load, ridgefill_fill  # noqa: E402
from late_layer_kv_gb300 import ridgefill as rb  # noqa: E402


def _both(shape, seed, rows_per_chunk=0):
    d = to_cuda(fill_inputs(shape, seed=seed))
    kw = dict(head_dim=shape.head_dim, rope_theta=shape.rope_theta, rms_eps=shape.rms_eps)
    K1, V1 = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
    ridgefill_fill(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], K1, V1, **kw)
    K2, V2 = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
    args = rb.fill_args(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], K2, V2,
                        rows_per_chunk=rows_per_chunk, **kw)
    lib = load()
    lib.ridgefill_fill_noalloc.argtypes = [ctypes.POINTER(rb.FillArgs), ctypes.c_void_p]
    lib.ridgefill_fill_noalloc.restype = ctypes.c_int
    st = lib.ridgefill_fill_noalloc(ctypes.byref(args), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.ridgefill_last_error().decode()
    torch.cuda.synchronize()
    assert device_error() == 0
    return (K1, V1), (K2, V2)


def test_noalloc_matches_workspace_fill_on_two_calls():
    # first call: 20 layers x 4096 -> scratch holds 384-row chunks, 3000 rows -> 8 chunks
    big = FillShape("noalloc_a", d=4096, n_layers=20, n_kv=8, head_dim=128, rope_theta=5e5,
                    rms_eps=1e-6, N=3000 + 512, T=512)
    # second call: another shape and seed through the same (now dirty) scratch
    small = FillShape("noalloc_b", d=256, n_layers=6, n_kv=2, head_dim=64, rope_theta=1e4,
                      rms_eps=1e-6, N=700, T=64)
    for shape, seed, rpc in ((big, 21, 0), (small, 22, 256)):
        (K1, V1), (K2, V2) = _both(shape, seed, rpc)
        rows = shape.rows
        # the per-row arithmetic does not depend on the chunking, so the two agree bit for
        # bit; any difference would be left over from the shared array's previous contents
        assert torch.equal(K2[:, :, :rows], K1[:, :, :rows]), f"{shape.name}: K differs"
        assert torch.equal(V2[:, :, :rows], V1[:, :, :rows]), f"{shape.name}: V differs"
        assert bool((K2[:, :, rows:] == SENTINEL).all()) and bool((V2[:, :, rows:] == SENTINEL).all())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = load()
    a = rb.FillArgs(400, 8192, 8192, 8, 128, 0, 1000, 0, 2048, 0, 1e4, 1e-6)
    lib.ridgefill_fill_noalloc.argtypes = [ctypes.POINTER(rb.FillArgs), ctypes.c_void_p]
    lib.ridgefill_fill_noalloc.restype = ctypes.c_int
    assert lib.ridgefill_fill_noalloc(ctypes.byref(a), None) == 8
    assert b"static scratch" in lib.ridgefill_last_error()
