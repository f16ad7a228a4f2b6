"""GPU parity of exact prefix rows (section 2.4) and of rho and the terminal-state
correction (section 2.3) against the f64 oracle.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
section 2.4 (a chosen subset of prefix rows runs every layer exactly) and
section 2.3 (rho: the share of the state that still comes from filled rows;
the state gets rho * Delta M once at the end of the prefix).
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import (WORKLOADS, FillShape, GdnShape, exact_rows, fill_inputs, gdn_inputs,
                       to_f64, true_inputs)
from tests._fill_helpers import SENTINEL, compare, new_cache, oracle_inputs, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import device_error, ridgefill_fill, ridgefill_fill_gdn  # noqa: E402

# rho is a ratio of sums of gate products; the gates come from bf16 inputs and
# projections (logit error ~2^-8 relative), so rho agrees to a few 1e-3 absolute.
RHO_ATOL = 5e-3


def _filled(n, exact):
    keep = np.ones(n, bool)
    keep[exact.numpy()] = False
    return torch.from_numpy(np.nonzero(keep)[0].astype(np.int32))


def _attn_fill(shape, d, Kc, Vc, pos0=0, row_idx=None, rows_per_chunk=0):
    ridgefill_fill(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                   head_dim=shape.head_dim, rope_theta=shape.rope_theta, rms_eps=shape.rms_eps,
                   pos0=pos0, rows_per_chunk=rows_per_chunk,
                   row_idx=None if row_idx is None else row_idx.cuda())
    torch.cuda.synchronize()


@pytest.mark.parametrize("rows_per_chunk", [0, 128])
def test_attention_fill_skips_exact_rows(rows_per_chunk):
    shape = FillShape("ex_mid", d=512, n_layers=3, n_kv=4, head_dim=128, rope_theta=5e5,
                      rms_eps=1e-6, N=700 + 60, T=60)
    inp = fill_inputs(shape, seed=91)
    d = to_cuda(inp)
    pos0 = 37
    fill = _filled(shape.rows, exact_rows(shape.rows, 0.3, seed=91))
    cache_len = pos0 + shape.N
    Kc, Vc = new_cache(3, 4, cache_len, 128)
    _attn_fill(shape, d, Kc, Vc, pos0=pos0, row_idx=fill, rows_per_chunk=rows_per_chunk)
    assert device_error() == 0
    Kf, Vf = new_cache(3, 4, cache_len, 128)
    _attn_fill(shape, d, Kf, Vf, pos0=pos0)
    pos = pos0 + fill.long()
    # listed rows: bitwise the rows of the unmasked fill; every other position untouched
    assert torch.equal(Kc[:, :, pos], Kf[:, :, pos]) and torch.equal(Vc[:, :, pos], Vf[:, :, pos])
    mask = torch.ones(cache_len, dtype=torch.bool, device="cuda")
    mask[pos.cuda()] = False
    assert bool((Kc[:, :, mask] == SENTINEL).all()) and bool((Vc[:, :, mask] == SENTINEL).all())
    o = oracle_inputs(inp)
    fi = fill.numpy()
    K, V = oracle.fill_attention(o["H"][fi], pos0 + fi, o["A"], o["b"], o["g"], o["Wk"],
                                 o["Wv"], shape.rms_eps, shape.rope_theta, 4, 128)
    for l in range(3):
        compare(to_f64(Kc[l][:, pos]), K[l], f"K layer {l}")
        compare(to_f64(Vc[l][:, pos]), V[l], f"V layer {l}")


def test_attention_full_size_masked_fill_bitwise():
    shape = WORKLOADS["llama8b_16k"]
    inp = fill_inputs(shape, seed=92)
    d = to_cuda(inp)
    fill = _filled(shape.rows, exact_rows(shape.rows, 0.3, seed=92))
    Kc, Vc = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
    _attn_fill(shape, d, Kc, Vc, row_idx=fill)
    assert device_error() == 0
    Kf, Vf = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
    _attn_fill(shape, d, Kf, Vf)
    pos = fill.long().cuda()
    assert torch.equal(Kc[:, :, pos], Kf[:, :, pos]) and torch.equal(Vc[:, :, pos], Vf[:, :, pos])
    mask = torch.ones(shape.N, dtype=torch.bool, device="cuda")
    mask[pos] = False
    assert bool((Kc[:, :, mask] == SENTINEL).all()) and bool((Vc[:, :, mask] == SENTINEL).all())


def test_out_of_range_index_is_skipped_and_reported():
    shape = FillShape("ex_bad", d=256, n_layers=1, n_kv=2, head_dim=64, rope_theta=1e4,
                      rms_eps=1e-6, N=200, T=0)
    d = to_cuda(fill_inputs(shape, seed=93))
    idx = torch.tensor([0, 5, 199, 200, 7], dtype=torch.int32)  # 200 is outside H's 200 rows
    Kc, Vc = new_cache(1, 2, 256, 64)
    _attn_fill(shape, d, Kc, Vc, row_idx=idx)
    assert device_error() == 6
    for p in (0, 5, 199, 7):
        assert not bool((Kc[:, :, p] == SENTINEL).all())
    assert bool((Kc[:, :, 200:] == SENTINEL).all())


def _gdn_shape(N=300):
    return GdnShape("ex_gdn", d=256, layer_kinds=("gdn",) * 2, n_heads=8, d_k=128, d_v=128,
                    chunk=64, n_kv=2, head_dim=128, rope_theta=1e4, rms_eps=1e-6, N=N, T=0)


def _gdn(shape, inp, exact=None, X=None, rho=False, dM=None, rows_per_chunk=0):
    d = {k: v.cuda() for k, v in inp.items()}
    L, H = shape.n_gdn, shape.n_heads
    S = torch.full((L, H, 128, 128), float("nan"), device="cuda")
    r = torch.full((L, H), float("nan"), device="cuda") if rho else None
    ridgefill_fill_gdn(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], d["Wa"], d["Wb"], S,
                       n_heads=H, rms_eps=shape.rms_eps, rows_per_chunk=rows_per_chunk,
                       exact_idx=None if exact is None else exact.cuda(),
                       X_exact=None if X is None else X.cuda(), rho=r,
                       delta_M=None if dM is None else dM.cuda())
    torch.cuda.synchronize()
    assert device_error() == 0
    return S.cpu(), (None if r is None else r.cpu())


@pytest.mark.parametrize("rows_per_chunk", [0, 128])
def test_gdn_exact_rows_state_and_rho(rows_per_chunk):
    shape = _gdn_shape()
    inp = gdn_inputs(shape, seed=94, gate_scale=3.0)
    exact = exact_rows(shape.rows, 0.3, seed=94)
    X = true_inputs(2, len(exact), 256, seed=94)
    S, rho = _gdn(shape, inp, exact, X, rho=True, rows_per_chunk=rows_per_chunk)
    o = {k: to_f64(v) for k, v in inp.items()}
    ex = exact.numpy()
    ref = oracle.gdn_state(o["H"], o["A"], o["b"], o["g"], o["Wk"], o["Wv"], o["Wa"], o["Wb"],
                           shape.rms_eps, 8, 128, 128, exact_idx=ex, X_exact=to_f64(X))
    for l in range(2):
        for h in range(8):
            compare(S[l, h].double().numpy(), ref[l, h], f"S layer {l} head {h}")
    rref = oracle.gdn_rho(o["H"], o["A"], o["b"], o["g"], o["Wa"], shape.rms_eps, 8,
                          exact_idx=ex, X_exact=to_f64(X))
    assert np.ptp(rref) > 0.3  # heads whose filled share differs widely
    np.testing.assert_allclose(rho.double().numpy(), rref, rtol=0, atol=RHO_ATOL)


def test_gdn_rho_is_one_without_exact_rows_and_zero_without_rows():
    shape = _gdn_shape()
    inp = gdn_inputs(shape, seed=95)
    _, rho = _gdn(shape, inp, rho=True, rows_per_chunk=128)
    assert bool((rho == 1.0).all())
    shape0 = _gdn_shape(N=0)
    inp0 = gdn_inputs(shape0, seed=95)
    _, rho0 = _gdn(shape0, inp0, rho=True)
    assert bool((rho0 == 0.0).all())


def test_terminal_state_correction():
    shape = _gdn_shape()
    inp = gdn_inputs(shape, seed=96, gate_scale=3.0)
    exact = exact_rows(shape.rows, 0.25, seed=96)
    X = true_inputs(2, len(exact), 256, seed=96)
    dM = torch.randn(2, 8, 128, 128, generator=torch.Generator().manual_seed(96))
    S1, rho = _gdn(shape, inp, exact, X, rho=True)
    S2, rho2 = _gdn(shape, inp, exact, X, rho=True, dM=dM)
    assert torch.equal(rho, rho2)
    want = oracle.terminal_correction(S1.double().numpy(), rho.double().numpy(), dM.double().numpy())
    np.testing.assert_allclose(S2.double().numpy(), want, rtol=1e-6, atol=1e-6)


def test_gdn_all_rows_exact_and_int8_maps():
    """Every prefix row exact (no map GEMM at all) and exact rows with int8 maps (mapped
    in full, then overwritten) both follow the oracle."""
    shape = _gdn_shape(N=200)
    inp = gdn_inputs(shape, seed=97)
    o = {k: to_f64(v) for k, v in inp.items()}
    every = torch.arange(shape.rows, dtype=torch.int32)
    X = true_inputs(2, shape.rows, 256, seed=97)
    S, rho = _gdn(shape, inp, every, X, rho=True)
    ref = oracle.gdn_state(o["H"], o["A"], o["b"], o["g"], o["Wk"], o["Wv"], o["Wa"], o["Wb"],
                           shape.rms_eps, 8, 128, 128, exact_idx=every.numpy(), X_exact=to_f64(X))
    for l in range(2):
        for h in range(8):
            compare(S[l, h].double().numpy(), ref[l, h], f"S layer {l} head {h}")
    assert bool((rho == 0.0).all())

    from late_layer_kv_gb300 import ridgefill_quantize_maps
    exact = exact_rows(shape.rows, 0.3, seed=97)
    Xe = true_inputs(2, len(exact), 256, seed=98)
    d = {k: v.cuda() for k, v in inp.items()}
    q, s = ridgefill_quantize_maps(d["A"])
    out = []
    for A, A_scale in ((q, s), (None, None)):
        if A is None:  # bf16 maps equal to bf16(q * s), compacted path
            w = q.cpu().float().reshape(2, 256, 2, 128) * s.cpu().float().transpose(1, 2)[..., None]
            A = w.reshape(2, 256, 256).to(torch.bfloat16).cuda()
        St = torch.empty((2, 8, 128, 128), device="cuda")
        ridgefill_fill_gdn(d["H"], A, d["b"], d["g"], d["Wk"], d["Wv"], d["Wa"], d["Wb"], St,
                           n_heads=8, rms_eps=shape.rms_eps, exact_idx=exact.cuda(),
                           X_exact=Xe.cuda(), A_scale=A_scale)
        out.append(St)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(out[0], out[1])  # full-map-then-overwrite == compacted, bit for bit
