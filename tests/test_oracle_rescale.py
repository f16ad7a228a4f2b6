"""Pins of the oracle's value/key rescale (section 2.3 "Value rescale", section 6.6).

Each test fixes the scale by a property of the definition, not by re-evaluating it:
exact prediction gives 1, sign flips and positive rescalings of the true inputs
give 1 (the norm removes them), a hand-built two-row case gives a known mean of
ratios, and a brute-force loop over rows and heads matches on a small case.
"""
import numpy as np

import oracle


def _case(seed=0, L=2, d_in=12, d_out=16, n_kv=2, hd=4, c=5):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((c, d_in))
    A = rng.standard_normal((L, d_out, d_in)) / np.sqrt(d_in)
    b = rng.standard_normal((L, d_out))
    g = 1 + 0.1 * rng.standard_normal((L, d_out))
    W = rng.standard_normal((L, n_kv * hd, d_out)) / np.sqrt(d_out)
    return H, A, b, g, W, n_kv, hd


def test_exact_prediction_gives_unit_scale():
    H, A, b, g, W, n_kv, hd = _case()
    X = np.stack([H @ A[l].T + b[l] for l in range(A.shape[0])])
    s = oracle.kv_rescale(H, X, A, b, g, W, 1e-6, n_kv, hd)
    np.testing.assert_allclose(s, 1.0, rtol=1e-12)


def test_sign_and_positive_scale_of_true_input_cancel():
    # RMSNorm(-x) = -RMSNorm(x) and RMSNorm(c x) = RMSNorm(x) (eps = 0): norms unchanged
    H, A, b, g, W, n_kv, hd = _case(1)
    X = np.stack([H @ A[l].T + b[l] for l in range(A.shape[0])])
    X *= np.array([-3.0, 0.25])[:, None, None]
    s = oracle.kv_rescale(H, X, A, b, g, W, 0.0, n_kv, hd)
    np.testing.assert_allclose(s, 1.0, rtol=1e-12)


def test_hand_built_mean_of_ratios():
    # one layer, d = 2, unit gain, W = identity (one head of width 2), eps = 0:
    # RMSNorm maps a row x to x / sqrt(mean(x^2)); its norm is sqrt(2) for any x != 0,
    # so build the ratio through W instead: W = diag(1, 0) keeps |x_0| / rms(x)
    H = np.array([[1.0, 0.0], [0.0, 1.0]])
    A = np.eye(2)[None]
    b = np.zeros((1, 2))
    g = np.ones((1, 2))
    W = np.diag([1.0, 0.0])[None]
    # predicted rows (1, 0) and (0, 1): |u_0| = sqrt(2) and 0 (left out)
    # true rows (1, 1) and (3, 4): |u_0| = 1 and 3 / sqrt(12.5)
    X = np.array([[[1.0, 1.0], [3.0, 4.0]]])
    s = oracle.kv_rescale(H, X, A, b, g, W, 0.0, 1, 2)
    assert abs(s[0, 0] - 1.0 / np.sqrt(2.0)) < 1e-15  # only row 0 counts: 1 / sqrt(2)
    # swap the prediction so both rows count
    H2 = np.array([[1.0, 0.0], [1.0, 0.0]])
    s2 = oracle.kv_rescale(H2, X, A, b, g, W, 0.0, 1, 2)
    want = 0.5 * (1.0 / np.sqrt(2.0) + (3.0 / np.sqrt(12.5)) / np.sqrt(2.0))
    assert abs(s2[0, 0] - want) < 1e-15


def test_brute_force_rows_and_heads():
    H, A, b, g, W, n_kv, hd = _case(2, L=2, n_kv=3, hd=4, c=6)
    rng = np.random.default_rng(9)
    X = rng.standard_normal((2, 6, 16))
    eps = 1e-3
    got = oracle.kv_rescale(H, X, A, b, g, W, eps, n_kv, hd)
    for l in range(2):
        for h in range(n_kv):
            ratios = []
            for r in range(6):
                def proj(x):
                    ms = sum(v * v for v in x) / len(x)
                    u = [x[j] / (ms + eps) ** 0.5 * g[l][j] for j in range(len(x))]
                    return [sum(W[l][h * hd + i][j] * u[j] for j in range(len(u))) for i in range(hd)]
                pred_x = [sum(A[l][o][k] * H[r][k] for k in range(H.shape[1])) + b[l][o] for o in range(16)]
                np_ = sum(v * v for v in proj(pred_x)) ** 0.5
                nt = sum(v * v for v in proj(list(X[l][r]))) ** 0.5
                ratios.append(nt / np_)
            assert abs(got[l, h] - sum(ratios) / len(ratios)) < 1e-12
