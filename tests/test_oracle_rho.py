"""Pins of the oracle's exact prefix rows and terminal-state correction.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
section 2.3 (terminal-state correction: rho, the share of the state that still
comes from filled rows; Figure 4) and section 2.4 (exact prefix rows).
"""
import json
import os

import numpy as np

import oracle
from synthetic import GdnShape, gdn_inputs, to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_figure4_printed_shares_with_a_row_mask():
    with open(os.path.join(GOLDEN, "figure4_gate_share.json")) as f:
        gd = json.load(f)
    rows, tail = gd["rows"], gd["tail"]
    filled = np.arange(rows) < rows - tail
    for c in gd["cases"]:
        rho = oracle.filled_share(np.full(rows, c["gate"]), filled)
        assert abs(rho - c["printed_share"]) <= c["printed_tolerance"], (c, rho)


def test_closed_forms():
    g, n = 0.93, 40
    even = np.arange(n) % 2 == 0  # weights g^(n-1-t): the even rows carry g, g^3, ...
    np.testing.assert_allclose(oracle.filled_share(np.full(n, g), even), g / (1 + g), rtol=1e-13)
    mask = np.random.default_rng(0).random(n) < 0.4
    assert oracle.filled_share(np.ones(n), mask) == mask.sum() / n
    assert oracle.filled_share(np.full(n, g), np.ones(n, bool)) == 1.0
    assert oracle.filled_share(np.full(n, g), np.zeros(n, bool)) == 0.0


def test_brute_force_products():
    rng = np.random.default_rng(1)
    for _ in range(5):
        n = int(rng.integers(1, 12))
        a = [float(x) for x in rng.uniform(0.2, 1.0, n)]
        f = [bool(x) for x in rng.random(n) < 0.5]
        num = den = 0.0
        for t in range(n):
            w = 1.0
            for s in range(t + 1, n):
                w *= a[s]
            den += w
            num += w if f[t] else 0.0
        np.testing.assert_allclose(oracle.filled_share(a, f), num / den, rtol=1e-14)


def test_rho_removes_a_common_shift_exactly():
    """The property section 2.3 states for the simplified model without the
    erase term: if every filled row's update is shifted by the same delta, the
    filled state differs from the exact one by rho times the difference with
    every row filled."""
    rng = np.random.default_rng(2)
    n, shape = 60, (3, 4)
    a = rng.uniform(0.9, 1.0, n)
    U = rng.standard_normal((n,) + shape)
    delta = rng.standard_normal(shape)
    filled = rng.random(n) < 0.7

    def run(shifted):
        S = np.zeros(shape)
        for t in range(n):
            S = a[t] * S + U[t] + (delta if shifted[t] else 0)
        return S

    exact = run(np.zeros(n, bool))
    diff_masked = run(filled) - exact
    diff_all = run(np.ones(n, bool)) - exact
    np.testing.assert_allclose(diff_masked, oracle.filled_share(a, filled) * diff_all, rtol=1e-12)


def _small():
    shape = GdnShape("rho_small", d=64, layer_kinds=("gdn",) * 2, n_heads=2, d_k=4, d_v=3,
                     chunk=64, n_kv=1, head_dim=64, rope_theta=1e4, rms_eps=1e-6, N=30, T=0)
    return shape, {k: to_f64(v) for k, v in gdn_inputs(shape, seed=5).items()}


def _args(o):
    return (o["H"], o["A"], o["b"], o["g"], o["Wk"], o["Wv"], o["Wa"], o["Wb"])


def test_exact_rows_equal_to_predictions_change_nothing():
    shape, o = _small()
    idx = np.array([3, 4, 17, 29])
    X = np.stack([oracle.map_apply(o["H"][idx], o["A"][l], o["b"][l]) for l in range(2)])
    base = oracle.gdn_state(*_args(o), shape.rms_eps, 2, 4, 3)
    got = oracle.gdn_state(*_args(o), shape.rms_eps, 2, 4, 3, exact_idx=idx, X_exact=X)
    np.testing.assert_allclose(got, base, rtol=1e-13, atol=1e-15)
    rho = oracle.gdn_rho(o["H"], o["A"], o["b"], o["g"], o["Wa"], shape.rms_eps, 2,
                         exact_idx=idx, X_exact=X)
    assert rho.shape == (2, 2) and np.all((rho > 0) & (rho < 1))


def test_exact_rows_enter_in_prompt_order():
    """Exact rows at the end: the state equals the filled rows' state carried on
    through the exact rows' own updates."""
    shape, o = _small()
    idx = np.arange(24, 30)
    X = np.random.default_rng(6).standard_normal((2, 6, 64)) * 3
    got = oracle.gdn_state(*_args(o), shape.rms_eps, 2, 4, 3, exact_idx=idx, X_exact=X)
    for l in range(2):
        xf = oracle.map_apply(o["H"][:24], o["A"][l], o["b"][l])
        k, v, a, b = oracle.gdn_projections(xf, o["g"][l], o["Wk"][l], o["Wv"][l], o["Wa"][l],
                                            o["Wb"][l], shape.rms_eps, 2, 4, 3)
        S = oracle.gdn_recurrence(k, v, a, b)
        k, v, a, b = oracle.gdn_projections(X[l], o["g"][l], o["Wk"][l], o["Wv"][l], o["Wa"][l],
                                            o["Wb"][l], shape.rms_eps, 2, 4, 3)
        np.testing.assert_allclose(got[l], oracle.gdn_recurrence(k, v, a, b, S), rtol=1e-12)


def test_rho_without_exact_rows_is_one_and_correction_is_linear():
    shape, o = _small()
    rho = oracle.gdn_rho(o["H"], o["A"], o["b"], o["g"], o["Wa"], shape.rms_eps, 2)
    np.testing.assert_allclose(rho, 1.0, rtol=0, atol=1e-15)
    rng = np.random.default_rng(7)
    S, dM = rng.standard_normal((2, 2, 3, 4)), rng.standard_normal((2, 2, 3, 4))
    np.testing.assert_array_equal(oracle.terminal_correction(S, np.zeros((2, 2)), dM), S)
    r = rng.random((2, 2))
    np.testing.assert_allclose(oracle.terminal_correction(S, r, dM) - S,
                               r[:, :, None, None] * dM, rtol=1e-14)
