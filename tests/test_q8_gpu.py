"""GPU parity of the int8 map path: ridgefill_quantize_maps against the oracle's
codes, and fills that read int8 maps against the oracle (maps q * s) and,
bitwise, against the bf16 path given the maps bf16(q * s).

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
section 2.2 ("Size and cost": int8 with one scale per 128 weights of each row)
and section 4.2.
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import WORKLOADS, FillShape, GdnShape, fill_inputs, gdn_inputs, tail_inputs, to_f64
from tests._fill_helpers import compare, new_cache, oracle_inputs, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import (  # noqa: E402
    RF_RESCALE_VALUES, device_error, ridgefill_fill, ridgefill_fill_gdn, ridgefill_quantize_maps,
    ridgefill_rescale)


def _rowmajor(s):
    """Group-major scales [L, G, d_out] as [L, d_out, G] (the oracle's layout)."""
    return s.transpose(1, 2).contiguous()


def _bf16_of_codes(q, s):
    """bf16(q * s) per weight (q * s is exact in f32), as CPU bf16."""
    L, d_out, d_in = q.shape
    w = q.float().reshape(L, d_out, d_in // 128, 128) * _rowmajor(s).float()[..., None]
    return w.reshape(L, d_out, d_in).to(torch.bfloat16)


def _quantize(A):
    q, s = ridgefill_quantize_maps(A.cuda())
    torch.cuda.synchronize()
    assert device_error() == 0
    return q.cpu(), s.cpu()


@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_quantizer_bitwise_equals_oracle(src):
    g = torch.Generator().manual_seed(5)
    A = torch.randn(3, 200, 640, generator=g) * torch.exp(torch.randn(3, 200, 1, generator=g))
    A[0, 7, 128:256] = 0.0                      # a zero group
    A[1, 3, :128] = torch.arange(128) - 64.0     # exact integers, a tie-rich group
    A[2, 5, 256:384] = 1e-30                     # tiny but normal
    A = A if src == "f32" else A.bfloat16()
    q, s = _quantize(A)
    q_ref, s_ref = oracle.quantize_map(A.float().numpy())
    assert np.array_equal(q.numpy(), q_ref)
    assert np.array_equal(_rowmajor(s).float().numpy(), s_ref)


def _fill(shape, d, A, A_scale=None, host=False, rows_per_chunk=0, group=0):
    Kc, Vc = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
    if host:
        A = A.cpu().pin_memory()
        A_scale = None if A_scale is None else A_scale.cpu().pin_memory()
    ridgefill_fill(d["H"], A, d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc, head_dim=shape.head_dim,
                   rope_theta=shape.rope_theta, rms_eps=shape.rms_eps, A_scale=A_scale,
                   rows_per_chunk=rows_per_chunk, q8_group_layers=group)
    torch.cuda.synchronize()
    assert device_error() == 0
    return Kc, Vc


@pytest.mark.parametrize("shape", [
    WORKLOADS["tiny_d256"],
    # d_out = 384: 128-column map tiles (64 rows of B per CTA); 333 rows: ragged, odd row tiles
    FillShape("q8_narrow", d=384, n_layers=3, n_kv=2, head_dim=128, rope_theta=5e5,
              rms_eps=1e-6, N=333 + 40, T=40),
])
def test_int8_fill_matches_oracle_and_bf16_path(shape):
    inp = fill_inputs(shape, seed=81)
    d = to_cuda(inp)
    q, s = ridgefill_quantize_maps(d["A"])
    K8, V8 = _fill(shape, d, q, s)
    # the bf16 path on the maps bf16(q * s) takes the same bits through the same MMAs
    Kb, Vb = _fill(shape, d, _bf16_of_codes(q.cpu(), s.cpu()).cuda())
    assert torch.equal(K8, Kb) and torch.equal(V8, Vb)
    o = oracle_inputs(inp)
    Aq = oracle.dequantize_map(q.cpu().numpy(), _rowmajor(s.cpu()).float().numpy())
    rows = shape.rows
    K, V = oracle.fill_attention(o["H"], np.arange(rows), Aq, o["b"], o["g"], o["Wk"], o["Wv"],
                                 shape.rms_eps, shape.rope_theta, shape.n_kv, shape.head_dim)
    for l in range(shape.n_layers):
        compare(to_f64(K8[l, :, :rows]), K[l], f"K layer {l}")
        compare(to_f64(V8[l, :, :rows]), V[l], f"V layer {l}")


def test_int8_host_maps_bitwise_equal_resident():
    shape = FillShape("q8_host", d=512, n_layers=5, n_kv=4, head_dim=128, rope_theta=5e5,
                      rms_eps=1e-6, N=640, T=100)
    d = to_cuda(fill_inputs(shape, seed=82))
    q, s = ridgefill_quantize_maps(d["A"])
    K1, V1 = _fill(shape, d, q, s)
    K2, V2 = _fill(shape, d, q, s, host=True)
    K3, V3 = _fill(shape, d, q, s, host=True, rows_per_chunk=256)
    assert torch.equal(K1, K2) and torch.equal(V1, V2)
    assert torch.equal(K1, K3) and torch.equal(V1, V3)


def test_int8_full_size_bitwise_equal_bf16_path():
    shape = WORKLOADS["llama8b_16k"]
    inp = fill_inputs(shape, seed=83, rows=4096)
    d = to_cuda(inp)
    q, s = ridgefill_quantize_maps(d["A"])
    sub = FillShape("q8_llama_rows4096", d=shape.d, n_layers=shape.n_layers, n_kv=shape.n_kv,
                    head_dim=shape.head_dim, rope_theta=shape.rope_theta, rms_eps=shape.rms_eps,
                    N=4096, T=0)
    K8, V8 = _fill(sub, d, q, s)
    Kb, Vb = _fill(sub, d, _bf16_of_codes(q.cpu(), s.cpu()).cuda())
    assert torch.equal(K8, Kb) and torch.equal(V8, Vb)


def test_int8_gdn_and_rescale_bitwise_equal_bf16_path():
    gs = GdnShape("q8_gdn", d=256, layer_kinds=("gdn",) * 2, n_heads=8, d_k=128, d_v=128,
                  chunk=64, n_kv=2, head_dim=128, rope_theta=1e4, rms_eps=1e-6, N=300, T=0)
    gd = {k: v.cuda() for k, v in gdn_inputs(gs, seed=84).items()}
    q, s = ridgefill_quantize_maps(gd["A"])
    Ab = _bf16_of_codes(q.cpu(), s.cpu()).cuda()
    out = []
    for A, A_scale in ((q, s), (Ab, None)):
        S = torch.empty((2, 8, 128, 128), dtype=torch.float32, device="cuda")
        ridgefill_fill_gdn(gd["H"], A, gd["b"], gd["g"], gd["Wk"], gd["Wv"], gd["Wa"], gd["Wb"], S,
                           n_heads=8, rms_eps=gs.rms_eps, A_scale=A_scale)
        out.append(S)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(out[0], out[1])

    shape = WORKLOADS["tiny_d256"]
    d = to_cuda(fill_inputs(shape, seed=85))
    t = to_cuda(tail_inputs(shape, seed=85, c=100))
    q, s = ridgefill_quantize_maps(d["A"])
    Ab = _bf16_of_codes(q.cpu(), s.cpu()).cuda()
    scales = []
    for A, A_scale in ((q, s), (Ab, None)):
        Kc, Vc = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
        sc = torch.empty((shape.n_layers, shape.n_kv), device="cuda")
        ridgefill_rescale(t["H_tail"], t["X_true"], A, d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                          which=RF_RESCALE_VALUES, head_dim=shape.head_dim,
                          rms_eps=shape.rms_eps, rows=0, scale=sc, A_scale=A_scale)
        scales.append(sc)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(scales[0], scales[1])


def test_int8_layer_groups_bitwise_equal_in_gemm_conversion():
    """Resident int8 maps dequantised a few layers at a time ahead of the bf16 GEMM (the
    default groups of 4, and groups of 1, 2 and 5 over 6 layers, with a ragged last group)
    give bitwise the caches of the conversion inside the GEMM (q8_group_layers = -1), also
    over row chunks."""
    shape = FillShape("q8_groups", d=512, n_layers=6, n_kv=4, head_dim=128, rope_theta=5e5,
                      rms_eps=1e-6, N=700, T=100)
    d = to_cuda(fill_inputs(shape, seed=86))
    q, s = ridgefill_quantize_maps(d["A"])
    K0, V0 = _fill(shape, d, q, s, group=-1)
    for group, rpc in ((0, 0), (1, 0), (2, 256), (5, 0)):
        K, V = _fill(shape, d, q, s, rows_per_chunk=rpc, group=group)
        assert torch.equal(K, K0) and torch.equal(V, V0), f"group {group}, chunk {rpc}"


def test_int8_gdn_layer_groups_with_exact_rows():
    """GDN fill with resident int8 maps: the grouped dequantisation (which also lets the map
    GEMM skip the exact rows) gives bitwise the state and rho of the in-GEMM conversion."""
    from synthetic import exact_rows, true_inputs
    gs = GdnShape("q8_gdn_groups", d=256, layer_kinds=("gdn",) * 3, n_heads=8, d_k=128, d_v=128,
                  chunk=64, n_kv=2, head_dim=128, rope_theta=1e4, rms_eps=1e-6, N=400, T=0)
    gd = {k: v.cuda() for k, v in gdn_inputs(gs, seed=87).items()}
    q, s = ridgefill_quantize_maps(gd["A"])
    rows = gs.N - gs.T
    idx = exact_rows(rows, 0.3, seed=87).to(torch.int32).cuda()
    X = true_inputs(3, idx.numel(), 256, seed=87).cuda()
    out = []
    for group in (-1, 0, 2):
        S = torch.empty((3, 8, 128, 128), dtype=torch.float32, device="cuda")
        rho = torch.empty((3, 8), dtype=torch.float32, device="cuda")
        ridgefill_fill_gdn(gd["H"], q, gd["b"], gd["g"], gd["Wk"], gd["Wv"], gd["Wa"], gd["Wb"], S,
                           n_heads=8, rms_eps=gs.rms_eps, A_scale=s, exact_idx=idx, X_exact=X,
                           rho=rho, q8_group_layers=group)
        out.append((S, rho))
    torch.cuda.synchronize()
    assert device_error() == 0
    for S, rho in out[1:]:
        assert torch.equal(S, out[0][0]) and torch.equal(rho, out[0][1])

