"""Options of ridgefill_fill combined, each checked bitwise against a simpler call that
must give the same bits: int8 maps streamed from host memory with a row list and row
chunks; a host split state with int8 maps; per-head value/key scales with a row list;
the no-allocation entry point with int8 maps.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill", sections
2.2 ("Size and cost"), 2.3 (value rescale), 2.4 (exact prefix rows) and 4.2 (maps in
VRAM or streamed from host, identical outputs).
"""
import ctypes

import numpy as np
import pytest
import torch

from synthetic import FillShape, exact_rows, fill_inputs
from tests._fill_helpers import SENTINEL, new_cache, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import (  # noqa: E402
    device_error, load, ridgefill_fill, ridgefill_quantize_maps)
from late_layer_kv_gb300 import ridgefill as rb  # noqa: E402

SHAPE = FillShape("combo", d=512, n_layers=3, n_kv=4, head_dim=128, rope_theta=5e5,
                  rms_eps=1e-6, N=5000 + 90, T=90)


def _kw():
    return dict(head_dim=SHAPE.head_dim, rope_theta=SHAPE.rope_theta, rms_eps=SHAPE.rms_eps)


def _fill(d, H, A, **kw):
    Kc, Vc = new_cache(SHAPE.n_layers, SHAPE.n_kv, SHAPE.N, SHAPE.head_dim)
    ridgefill_fill(H, A, d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc, **_kw(), **kw)
    torch.cuda.synchronize()
    assert device_error() == 0
    return Kc, Vc


def _filled(n, exact):
    keep = np.ones(n, bool)
    keep[exact.numpy()] = False
    return torch.from_numpy(np.nonzero(keep)[0].astype(np.int32)).cuda()


def _same(a, b):
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_int8_host_maps_row_list_and_chunks():
    d = to_cuda(fill_inputs(SHAPE, seed=101))
    q, s = ridgefill_quantize_maps(d["A"])
    idx = _filled(SHAPE.rows, exact_rows(SHAPE.rows, 0.25, seed=101))
    ref = _fill(d, d["H"], q, A_scale=s, row_idx=idx)
    got = _fill(d, d["H"], q.cpu().pin_memory(), A_scale=s.cpu().pin_memory(), row_idx=idx,
                rows_per_chunk=1024)
    _same(ref, got)
    assert bool((got[0][:, :, SHAPE.rows:] == SENTINEL).all())


def test_host_split_state_with_int8_maps():
    inp = fill_inputs(SHAPE, seed=102)
    d = to_cuda(inp)
    q, s = ridgefill_quantize_maps(d["A"])
    _same(_fill(d, d["H"], q, A_scale=s), _fill(d, inp["H"].pin_memory(), q, A_scale=s))


def test_value_scales_with_row_list():
    d = to_cuda(fill_inputs(SHAPE, seed=103))
    idx = _filled(SHAPE.rows, exact_rows(SHAPE.rows, 0.3, seed=103))
    g = torch.Generator().manual_seed(103)
    vs = (0.5 + torch.rand(SHAPE.n_layers, SHAPE.n_kv, generator=g)).cuda()
    ks = (0.5 + torch.rand(SHAPE.n_layers, SHAPE.n_kv, generator=g)).cuda()
    full = _fill(d, d["H"], d["A"], v_scale=vs, k_scale=ks)
    part = _fill(d, d["H"], d["A"], v_scale=vs, k_scale=ks, row_idx=idx, rows_per_chunk=512)
    pos = idx.long()
    assert torch.equal(full[0][:, :, pos], part[0][:, :, pos])
    assert torch.equal(full[1][:, :, pos], part[1][:, :, pos])
    # the scales really act: one head's values differ from the unscaled fill
    plain = _fill(d, d["H"], d["A"])
    assert not torch.equal(plain[1][:, :, pos], part[1][:, :, pos])


def test_noalloc_with_int8_maps():
    d = to_cuda(fill_inputs(SHAPE, seed=104))
    q, s = ridgefill_quantize_maps(d["A"])
    ref = _fill(d, d["H"], q, A_scale=s)
    K2, V2 = new_cache(SHAPE.n_layers, SHAPE.n_kv, SHAPE.N, SHAPE.head_dim)
    args = rb.fill_args(d["H"], q, d["b"], d["g"], d["Wk"], d["Wv"], K2, V2, A_scale=s, **_kw())
    lib = load()
    lib.ridgefill_fill_noalloc.argtypes = [ctypes.POINTER(rb.FillArgs), ctypes.c_void_p]
    lib.ridgefill_fill_noalloc.restype = ctypes.c_int
    st = lib.ridgefill_fill_noalloc(ctypes.byref(args), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.ridgefill_last_error().decode()
    torch.cuda.synchronize()
    assert device_error() == 0
    _same(ref, (K2, V2))
