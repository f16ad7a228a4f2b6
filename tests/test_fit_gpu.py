"""GPU parity of ridgefill_fit (running sums and closed-form solve) against the f64
oracle.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
section 2.2 ("The ridge map", "Fitting": running sums one document at a time
give the all-rows solve, "The penalty").
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import WORKLOADS, calibration, calibration_device, fill_inputs, to_f64
from tests._fill_helpers import compare, new_cache

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import (FitSums, device_error, ridgefill_fill,  # noqa: E402
                                 ridgefill_fit_accumulate, ridgefill_fit_solve)

W_REL_FRO = 1e-3  # fitted maps: relative Frobenius error against the f64 solve


def _rel(a, b):
    return np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b)


def _gpu_fit(X, Y, lam, batches=(None,)):
    L, n, d_out = Y.shape
    d_in = X.shape[1]
    sums = FitSums(L, d_in, d_out)
    Xd, Yd = X.cuda(), Y.cuda()
    bounds = [0] + [b for b in batches if b is not None] + [n]
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        ridgefill_fit_accumulate(sums, Xd[lo:hi].contiguous(), Yd[:, lo:hi].contiguous())
    A32 = torch.empty((L, d_out, d_in), dtype=torch.float32, device="cuda")
    A16 = torch.empty((L, d_out, d_in), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((L, d_out), dtype=torch.float32, device="cuda")
    alpha = torch.zeros(1, dtype=torch.float64, device="cuda")
    ridgefill_fit_solve(sums, lam, A_out=A16, A_out_f32=A32, b_out=b, alpha_out=alpha)
    torch.cuda.synchronize()
    assert device_error() == 0
    return sums, A32.cpu().double().numpy(), A16, b.cpu().double().numpy(), float(alpha.item())


# Gram tiles: 256 columns (d = 256, and small products at d = 512 and 1024); 512 columns on
# clusters of two CTA pairs once the tiles fill eight waves of pairs (d = 1024 with 201 layers
# of d_out = 384: an odd row-tile count leaves the last pair of the last cluster half empty);
# 777 and 300 rows end in ragged 64-row blocks
@pytest.mark.parametrize("d,L,n,d_out,cut", [(256, 3, 1000, 256, 600), (1024, 2, 777, 1024, 320),
                                             (512, 1, 300, 384, 128), (1024, 201, 300, 384, 100)])
def test_sums_match_oracle_and_split_batches(d, L, n, d_out, cut):
    cal = calibration(d=d, n_layers=L, n=n, seed=40 + d)
    X, Y = cal["X"], cal["Y"][:, :, :d_out].contiguous()
    sums, *_ = _gpu_fit(X, Y, 1e-3, batches=(cut,))
    n, sx, sy, G, C = oracle.fit_sums(to_f64(X), to_f64(Y))
    assert float(sums.count.item()) == n
    np.testing.assert_allclose(sums.sx.cpu().numpy(), sx, rtol=2e-5, atol=2e-5 * np.abs(sx).max())
    np.testing.assert_allclose(sums.sy.cpu().numpy(), sy, rtol=2e-5, atol=2e-5 * np.abs(sy).max())
    # f32 sums of up to 600 exact products per batch: relative error ~ sqrt(n) u, n u = 6e-5 at worst
    assert _rel(sums.G.cpu().numpy(), G) < 2e-5
    Cg = sums.C.cpu().numpy()                       # [L, d_out, d_in] = Y_l^T X
    Co = C.reshape(d, L, d_out).transpose(1, 2, 0)  # oracle [d_in, L*d_out] -> [L, d_out, d_in]
    assert _rel(Cg, Co) < 2e-5


def test_tiny_batches_add_exactly_what_they_hold():
    """Batches of 0, 1, 63 and 65 rows (none, part of one 64-row block, one row past it) on
    the clustered 512-column Gram path: the sums are those of the rows given."""
    cal = calibration(d=1024, n_layers=201, n=129, seed=47)
    X, Y = cal["X"], cal["Y"][:, :, :384].contiguous()
    sums = FitSums(201, 1024, 384)
    Xd, Yd = X.cuda(), Y.cuda()
    bounds = [0, 0, 1, 64, 129]  # an empty batch, then 1, 63 and 65 rows
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        ridgefill_fit_accumulate(sums, Xd[lo:hi].contiguous(), Yd[:, lo:hi].contiguous())
    torch.cuda.synchronize()
    assert device_error() == 0
    n, sx, sy, G, C = oracle.fit_sums(to_f64(X), to_f64(Y))
    assert float(sums.count.item()) == n
    np.testing.assert_allclose(sums.sx.cpu().numpy(), sx, rtol=1e-6, atol=1e-6 * np.abs(sx).max())
    np.testing.assert_allclose(sums.sy.cpu().numpy(), sy, rtol=1e-6, atol=1e-6 * np.abs(sy).max())
    assert _rel(sums.G.cpu().numpy(), G) < 1e-5
    assert _rel(sums.C.cpu().numpy(), C.reshape(1024, 201, 384).transpose(1, 2, 0)) < 1e-5


def test_full_size_sums_sampled():
    """The fit workload at full size (d = 4096, 20 layers, 65,536 calibration rows), on the
    clustered Gram path the bench times: the sums of 64 sampled X columns and 64 sampled
    output channels of every layer against the oracle's sums of those columns over every
    row."""
    shape = WORKLOADS["hostmaps_16k"]
    d, L, n = shape.d, shape.n_layers, shape.calib_rows
    cal = calibration_device(d, L, n, seed=1003, device="cuda")
    X, Y = cal["X"], cal["Y"]
    sums = FitSums(L, d, d)
    ridgefill_fit_accumulate(sums, X, Y)
    torch.cuda.synchronize()
    assert device_error() == 0
    rng = np.random.default_rng(11)
    ci = np.sort(rng.choice(d, 64, replace=False))  # X columns
    co = np.sort(rng.choice(d, 64, replace=False))  # output channels of each layer
    ti, to = torch.from_numpy(ci).cuda(), torch.from_numpy(co).cuda()
    Xs = X[:, ti].cpu()
    Ys = Y[:, :, to].cpu()
    del X, Y, cal
    torch.cuda.empty_cache()
    nn, sx, sy, G, C = oracle.fit_sums(to_f64(Xs), to_f64(Ys))  # C: [64, L * 64]
    assert float(sums.count.item()) == nn == n
    Gg = sums.G[ti][:, ti].cpu().numpy()
    Cg = sums.C[:, to][:, :, ti].cpu().numpy()               # [L, 64 outputs, 64 inputs]
    Co = C.reshape(64, L, 64).transpose(1, 2, 0)
    # each entry is 4096 f32 accumulations of 16-product MMA steps: at most 4096 * 2^-24
    # = 2.4e-4 of its magnitude even if every rounding went the same way
    assert _rel(Gg, G) < 5e-4
    assert _rel(Cg, Co) < 5e-4
    np.testing.assert_allclose(sums.sx[ti].cpu().numpy(), sx, rtol=1e-6, atol=1e-6 * np.abs(sx).max())
    np.testing.assert_allclose(sums.sy[:, to].cpu().numpy(), sy, rtol=1e-6,
                               atol=1e-6 * np.abs(sy).max())


def test_full_size_fit_sampled():
    """The whole fit at full size (d = 4096, 20 layers, 65,536 rows: the clustered Gram, the
    blocked Cholesky and the split-bf16 solve the bench runs): eight output channels of the
    first and the last layer against the oracle's ridge fit of those channels.  A channel's
    map row and offset depend only on X and on its own column of Y, so the oracle fits the
    sampled columns alone."""
    shape = WORKLOADS["hostmaps_16k"]
    d, L, n = shape.d, shape.n_layers, shape.calib_rows
    cal = calibration_device(d, L, n, seed=1004, device="cuda")
    X, Y = cal["X"], cal["Y"]
    sums = FitSums(L, d, d)
    ridgefill_fit_accumulate(sums, X, Y)
    A32 = torch.empty((L, d, d), dtype=torch.float32, device="cuda")
    b = torch.empty((L, d), dtype=torch.float32, device="cuda")
    alpha = torch.zeros(1, dtype=torch.float64, device="cuda")
    ridgefill_fit_solve(sums, shape.lam, A_out_f32=A32, b_out=b, alpha_out=alpha)
    torch.cuda.synchronize()
    assert device_error() == 0
    js = torch.from_numpy(np.sort(np.random.default_rng(13).choice(d, 8, replace=False))).cuda()
    layers = torch.tensor([0, L - 1], device="cuda")
    Ys = Y[layers][:, :, js].cpu()
    Ag = A32[layers][:, js].cpu().double().numpy()   # [2, 8, d_in]
    bg = b[layers][:, js].cpu().double().numpy()
    Xh = X.cpu()
    del X, Y, cal, A32
    torch.cuda.empty_cache()
    Ao, bo, ao = oracle.ridge_fit(to_f64(Xh), to_f64(Ys), shape.lam)
    # alpha = lam tr(X~^T X~) / d_in takes the Gram diagonal, summed over the 65,536 rows of
    # the one batch in f32 on the tensor cores (4096 accumulation steps a sum; measured
    # 3e-4 low, against at most 4096 * 2^-23 = 4.9e-4 with every step truncated)
    assert abs(float(alpha.item()) - ao) <= 1e-3 * ao
    for i in range(2):
        assert _rel(Ag[i], Ao[i]) <= W_REL_FRO, f"layer {i}: {_rel(Ag[i], Ao[i]):.2e}"
        assert _rel(bg[i], bo[i]) <= W_REL_FRO


# d = 384 and 640 are not powers of two: the blocked inverse then merges a last,
# shorter block pair
@pytest.mark.parametrize("d,L,n,lam", [(256, 3, 1000, 1e-3), (512, 2, 4096, 3e-2),
                                       (384, 2, 2000, 1e-3), (640, 2, 3000, 1e-2)])
def test_solve_matches_closed_form(d, L, n, lam):
    cal = calibration(d=d, n_layers=L, n=n, seed=41 + d)
    X, Y = cal["X"], cal["Y"]
    _, A32, A16, b, alpha = _gpu_fit(X, Y, lam, batches=(n // 3,))
    Ao, bo, ao = oracle.ridge_fit(to_f64(X), to_f64(Y), lam)
    assert abs(alpha - ao) <= 1e-5 * ao
    for l in range(L):
        assert _rel(A32[l], Ao[l]) <= W_REL_FRO, f"layer {l}: {_rel(A32[l], Ao[l]):.2e}"
        assert _rel(b[l], bo[l]) <= W_REL_FRO
        # the bf16 output is the f32 output rounded
        np.testing.assert_array_equal(to_f64(A16[l]), to_f64(torch.from_numpy(A32[l]).float()
                                                            .to(torch.bfloat16)))


def test_solve_centres_sums_with_large_means():
    """Sums of columns whose means are 1,000 standard deviations from zero (and outputs 500
    from zero), built in f64 and handed to the solve directly: the centred Gram and
    cross terms cancel about 20 of the leading bits of every entry, which the solve's
    centring keeps (a plain f32 centring would leave errors of order 2^-3)."""
    rng = np.random.default_rng(47)
    d, L, n, lam = 256, 2, 3000, 1e-3
    X = rng.standard_normal((n, d))
    X[:, : d // 2] += 1000.0
    W = rng.standard_normal((L, d, d)) / np.sqrt(d)
    Y = np.einsum("nk,lko->lno", X - X.mean(axis=0), W) + 500.0 + 0.1 * rng.standard_normal((L, n, d))
    cnt, sx, sy, G, C = oracle.fit_sums(X, Y)
    sums = FitSums(L, d, d)
    sums.G.copy_(torch.from_numpy(G))
    sums.C.copy_(torch.from_numpy(C.T.reshape(L, d, d)))
    sums.sx.copy_(torch.from_numpy(sx))
    sums.sy.copy_(torch.from_numpy(sy))
    sums.count.fill_(float(cnt))
    A32 = torch.empty((L, d, d), dtype=torch.float32, device="cuda")
    b = torch.empty((L, d), dtype=torch.float32, device="cuda")
    ridgefill_fit_solve(sums, lam, A_out_f32=A32, b_out=b)
    torch.cuda.synchronize()
    assert device_error() == 0
    Ao, bo, _ = oracle.ridge_solve_from_sums(cnt, sx, sy, G, C, lam)
    A = A32.cpu().double().numpy()
    bg = b.cpu().double().numpy()
    mu_x = sx / cnt
    for l in range(L):
        assert _rel(A[l], Ao[l]) <= W_REL_FRO, f"layer {l}: {_rel(A[l], Ao[l]):.2e}"
        # b = mu_y - A mu_x: the map's error is carried by mu_x, whose entries are 1,000
        scale = np.linalg.norm(Ao[l]) * np.linalg.norm(mu_x) + np.linalg.norm(bo[l])
        assert np.linalg.norm(bg[l] - bo[l]) <= W_REL_FRO * scale


def test_batch_split_does_not_change_the_fit():
    cal = calibration(d=256, n_layers=2, n=2048, seed=43)
    _, A1, _, b1, _ = _gpu_fit(cal["X"], cal["Y"], 1e-3)
    _, A2, _, b2, _ = _gpu_fit(cal["X"], cal["Y"], 1e-3, batches=(64, 1000, 1999))
    # the sums differ only by f32 rounding inside each batch; the solve carries ~2^-16 of
    # each operand (three-term bf16 split), so two batchings agree to ~1e-5
    assert _rel(A2, A1) < 1e-4 and _rel(b2, b1) < 1e-4


def test_noise_free_recovers_generating_map():
    """Y = X M + c exactly (f64, then rounded to bf16 inputs) with a tiny penalty:
    the fit returns A = M^T and b = c up to the bf16 rounding of Y."""
    rng = np.random.default_rng(44)
    d, n = 256, 4096
    X = torch.from_numpy((rng.standard_normal((n, d)) * 2).astype(np.float32)).to(torch.bfloat16)
    M = (np.eye(d) + 0.1 * rng.standard_normal((d, d)) / 16).astype(np.float64)
    c = rng.standard_normal(d)
    Y = torch.from_numpy((to_f64(X) @ M + c).astype(np.float32)).to(torch.bfloat16)[None]
    _, A, _, b, _ = _gpu_fit(X, Y, 1e-9)
    Ao, bo, _ = oracle.ridge_fit(to_f64(X), to_f64(Y), 1e-9)
    assert _rel(A[0], Ao[0]) <= W_REL_FRO
    assert _rel(A[0], M.T) < 5e-3          # bf16 rounding of Y limits the recovery
    assert np.abs(b[0] - c).max() < 0.05


def test_tiny_fit_then_fill_end_to_end():
    """Config tiny_d256: fit six maps from 4,096 calibration rows, then fill 448 prefix
    rows with the fitted (bf16) maps; both steps against the oracle."""
    shape = WORKLOADS["tiny_d256"]
    cal = calibration(d=shape.d, n_layers=shape.n_layers, n=shape.calib_rows, seed=1000)
    _, A32, A16, b, _ = _gpu_fit(cal["X"], cal["Y"], shape.lam)
    Ao, bo, _ = oracle.ridge_fit(to_f64(cal["X"]), to_f64(cal["Y"]), shape.lam)
    assert _rel(A32, Ao) <= W_REL_FRO
    inp = fill_inputs(shape, seed=1000)
    inp["A"] = A16.cpu()
    inp["b"] = torch.from_numpy(b.astype(np.float32))
    d = {k: v.cuda() for k, v in inp.items()}
    Kc, Vc = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
    ridgefill_fill(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                   head_dim=shape.head_dim, rope_theta=shape.rope_theta, rms_eps=shape.rms_eps)
    torch.cuda.synchronize()
    o = {k: to_f64(v) for k, v in inp.items()}
    K, V = oracle.fill_attention(o["H"], np.arange(shape.rows), o["A"], o["b"], o["g"], o["Wk"],
                                 o["Wv"], shape.rms_eps, shape.rope_theta, shape.n_kv,
                                 shape.head_dim)
    for l in range(shape.n_layers):
        compare(to_f64(Kc[l, :, :shape.rows]), K[l], f"K layer {l}")
        compare(to_f64(Vc[l, :, :shape.rows]), V[l], f"V layer {l}")
