"""Pins of the oracle's ridge fit against what the paper and mathematics fix.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
section 2.2 (objective, closed form, running sums, penalty).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _data(n=200, d_in=6, d_out=5, L=2, seed=0, noise=0.1):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((n, d_in)) * np.exp(rng.standard_normal(d_in)) + rng.standard_normal(d_in)
    M = rng.standard_normal((L, d_out, d_in))
    c = rng.standard_normal((L, d_out))
    Y = np.einsum("loi,ni->lno", M, X) + c[:, None, :] + noise * rng.standard_normal((L, n, d_out))
    return X, Y, M, c


def test_objective_is_stationary():
    """Gradient of the printed objective sum ||x_l - (A x_S + b)||^2 + alpha ||A||_F^2
    vanishes at the returned (A, b); evaluated on the raw (uncentred) rows."""
    X, Y, _, _ = _data()
    A, b, alpha = oracle.ridge_fit(X, Y, lam=0.03)
    for l in range(Y.shape[0]):
        R = Y[l] - X @ A[l].T - b[l]                 # residual per token
        gA = -2.0 * R.T @ X + 2.0 * alpha * A[l]
        gb = -2.0 * R.sum(axis=0)
        scale = np.abs(R).sum() * np.abs(X).max()
        assert np.abs(gA).max() / scale < 1e-12
        assert np.abs(gb).max() / np.abs(R).sum() < 1e-12


def test_matches_augmented_least_squares():
    """Ridge = least squares on [X~; sqrt(alpha) I] (textbook identity), via lstsq."""
    X, Y, _, _ = _data(seed=1)
    A, b, alpha = oracle.ridge_fit(X, Y, lam=0.01)
    Xc = X - X.mean(0)
    d = X.shape[1]
    for l in range(Y.shape[0]):
        Yc = Y[l] - Y[l].mean(0)
        Xa = np.vstack([Xc, np.sqrt(alpha) * np.eye(d)])
        Ya = np.vstack([Yc, np.zeros((d, Y.shape[2]))])
        At, *_ = np.linalg.lstsq(Xa, Ya, rcond=None)
        np.testing.assert_allclose(A[l], At.T, rtol=1e-10, atol=1e-12)


def test_matches_sklearn_ridge():
    """scikit-learn's Ridge with intercept solves the same problem for a given alpha."""
    sk = pytest.importorskip("sklearn.linear_model")
    X, Y, _, _ = _data(seed=2, n=300)
    A, b, alpha = oracle.ridge_fit(X, Y, lam=0.05)
    for l in range(Y.shape[0]):
        m = sk.Ridge(alpha=alpha, fit_intercept=True, solver="cholesky").fit(X, Y[l])
        np.testing.assert_allclose(A[l], m.coef_, rtol=1e-8, atol=1e-10)
        np.testing.assert_allclose(b[l], m.intercept_, rtol=1e-8, atol=1e-10)


def test_penalty_definition_alpha():
    """alpha = lambda * tr(X~^T X~) / d_in, with X~ the centred split states."""
    X, Y, _, _ = _data(seed=3)
    _, _, alpha = oracle.ridge_fit(X, Y, lam=0.2)
    ss = sum(float(v - X[:, j].mean()) ** 2 for j in range(X.shape[1]) for v in X[:, j])
    assert abs(alpha - 0.2 * ss / X.shape[1]) < 1e-9 * alpha


def test_penalty_scale_invariance():
    """Scaling the split state by c leaves predictions unchanged: the penalty
    follows the input size, so one lambda means the same on every model."""
    X, Y, _, _ = _data(seed=4)
    A1, b1, _ = oracle.ridge_fit(X, Y, lam=0.03)
    A2, b2, _ = oracle.ridge_fit(7.5 * X, Y, lam=0.03)
    np.testing.assert_allclose(A2 * 7.5, A1, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(b2, b1, rtol=1e-9, atol=1e-12)


def test_noise_free_recovers_generating_map():
    X, Y, M, c = _data(seed=5, noise=0.0)
    A, b, _ = oracle.ridge_fit(X, Y, lam=1e-13)
    np.testing.assert_allclose(A, M, rtol=0, atol=1e-7)
    np.testing.assert_allclose(b, c, rtol=0, atol=1e-7)


def test_mean_residual_is_zero():
    """The offset makes the map right on average over the calibration rows."""
    X, Y, _, _ = _data(seed=6)
    A, b, _ = oracle.ridge_fit(X, Y, lam=0.5)
    for l in range(Y.shape[0]):
        r = (Y[l] - X @ A[l].T - b[l]).mean(axis=0)
        assert np.abs(r).max() < 1e-12 * np.abs(Y[l]).max()


def _frac_ridge_2x2(X, Y, lam):
    """Exact rational ridge for d_in = 2 by the adjugate formula (brute force)."""
    n = len(X)
    mx = [sum(r[j] for r in X) / n for j in range(2)]
    my = [sum(r[j] for r in Y) / n for j in range(len(Y[0]))]
    Xc = [[r[j] - mx[j] for j in range(2)] for r in X]
    Yc = [[r[j] - my[j] for j in range(len(my))] for r in Y]
    G = [[sum(Xc[t][i] * Xc[t][j] for t in range(n)) for j in range(2)] for i in range(2)]
    alpha = lam * (G[0][0] + G[1][1]) / 2
    a, bb, c, d = G[0][0] + alpha, G[0][1], G[1][0], G[1][1] + alpha
    det = a * d - bb * c
    inv = [[d / det, -bb / det], [-c / det, a / det]]
    A = []
    for o in range(len(my)):
        yx = [sum(Yc[t][o] * Xc[t][i] for t in range(n)) for i in range(2)]
        A.append([yx[0] * inv[0][j] + yx[1] * inv[1][j] for j in range(2)])
    b = [my[o] - (A[o][0] * mx[0] + A[o][1] * mx[1]) for o in range(len(my))]
    return A, b, alpha


def test_exact_rational_two_by_two():
    F = Fraction
    X = [[F(1), F(2)], [F(3), F(5)], [F(4), F(-1)]]
    Y = [[F(1), F(0)], [F(2), F(1)], [F(0), F(3)]]
    lam = F(1, 10)
    Ae, be, ae = _frac_ridge_2x2(X, Y, lam)
    A, b, alpha = oracle.ridge_fit(np.array(X, float), np.array([Y], float), lam=0.1)
    assert abs(alpha - float(ae)) < 1e-12
    np.testing.assert_allclose(A[0], np.array(Ae, float), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(b[0], np.array(be, float), rtol=1e-12, atol=1e-14)


def test_streaming_sums_equal_one_shot():
    """Running sums one document at a time give the all-rows solve (section 2.2)."""
    X, Y, _, _ = _data(seed=7, n=301)
    A, b, alpha = oracle.ridge_fit(X, Y, lam=0.03)
    parts = [(0, 50), (50, 51), (51, 200), (200, 301)]
    acc = None
    for lo, hi in parts:
        s = oracle.fit_sums(X[lo:hi], Y[:, lo:hi])
        acc = s if acc is None else tuple(x + y for x, y in zip(acc, s))
    A2, b2, a2 = oracle.ridge_solve_from_sums(*acc, lam=0.03)
    assert abs(a2 - alpha) < 1e-9 * alpha
    np.testing.assert_allclose(A2, A, rtol=1e-8, atol=1e-10)
    np.testing.assert_allclose(b2, b, rtol=1e-8, atol=1e-10)


def test_fit_sums_by_loops():
    X, Y, _, _ = _data(seed=8, n=9, d_in=3, d_out=2, L=2)
    n, sx, sy, G, C = oracle.fit_sums(X, Y)
    assert n == 9
    for i in range(3):
        assert abs(sx[i] - sum(X[t, i] for t in range(9))) < 1e-12
        for j in range(3):
            assert abs(G[i, j] - sum(X[t, i] * X[t, j] for t in range(9))) < 1e-11
        for l in range(2):
            for o in range(2):
                assert abs(C[i, l * 2 + o] - sum(X[t, i] * Y[l, t, o] for t in range(9))) < 1e-11
