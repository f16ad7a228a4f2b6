"""Pins of the oracle's Gated DeltaNet state fill and host arithmetic.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
section 2.3 (Gated DeltaNet layers, terminal-state correction, Figure 4) and
section 2.5 (compute ceiling).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rows, nh, dk, dv, seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((rows, nh, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((rows, nh, dv))
    a = 1 / (1 + np.exp(-rng.standard_normal((rows, nh))))
    b = 1 / (1 + np.exp(-rng.standard_normal((rows, nh))))
    return k, v, a, b


def test_literal_matrix_product_form():
    """Brute force with the explicit (I - beta k k^T) matrix product."""
    k, v, a, b = _rand(13, 2, 5, 3, 0)
    S = oracle.gdn_recurrence(k, v, a, b)
    for h in range(2):
        M = np.zeros((3, 5))
        for t in range(13):
            P = np.eye(5) - b[t, h] * np.outer(k[t, h], k[t, h])
            M = a[t, h] * (M @ P) + b[t, h] * np.outer(v[t, h], k[t, h])
        np.testing.assert_allclose(S[h], M, rtol=1e-12, atol=1e-13)


def test_single_step_from_zero():
    k, v, a, b = _rand(1, 3, 4, 6, 1)
    S = oracle.gdn_recurrence(k, v, a, b)
    for h in range(3):
        np.testing.assert_allclose(S[h], b[0, h] * np.outer(v[0, h], k[0, h]), rtol=1e-14)


def test_beta_zero_only_decays_initial_state():
    k, v, a, _ = _rand(20, 2, 4, 4, 2)
    S0 = np.random.default_rng(3).standard_normal((2, 4, 4))
    S = oracle.gdn_recurrence(k, v, a, np.zeros((20, 2)), S0)
    np.testing.assert_allclose(S, np.prod(a, axis=0)[:, None, None] * S0, rtol=1e-12)


def test_delta_rule_memory_with_orthonormal_keys():
    """alpha = beta = 1 and orthonormal keys: the state maps each written key to
    its value (the delta rule overwrites the association along k)."""
    dk = 8
    Q, _ = np.linalg.qr(np.random.default_rng(4).standard_normal((dk, dk)))
    k = Q.T[:6][:, None, :]                    # 6 orthonormal keys
    v = np.random.default_rng(5).standard_normal((6, 1, 3))
    S = oracle.gdn_recurrence(k, v, np.ones((6, 1)), np.ones((6, 1)),
                              np.random.default_rng(6).standard_normal((1, 3, dk)))
    for t in range(6):
        np.testing.assert_allclose(S[0] @ k[t, 0], v[t, 0], rtol=1e-12, atol=1e-12)


def test_rewrite_same_key_replaces_value():
    k = np.zeros((2, 1, 4)); k[:, 0, 1] = 1.0
    v = np.array([[[1.0, 2.0]], [[-3.0, 5.0]]])
    S = oracle.gdn_recurrence(k, v, np.ones((2, 1)), np.ones((2, 1)))
    np.testing.assert_allclose(S[0] @ k[0, 0], v[1, 0], rtol=1e-14)


def test_gdn_state_brute_force_tiny():
    """Projections + recurrence for d=6, 2 heads, by plain loops."""
    rng = np.random.default_rng(7)
    d, nh, dk, dv, rows = 6, 2, 3, 2, 5
    H = rng.standard_normal((rows, d))
    A = rng.standard_normal((1, d, d)); b = rng.standard_normal((1, d))
    g = 1 + 0.1 * rng.standard_normal((1, d))
    Wk = rng.standard_normal((1, nh * dk, d)); Wv = rng.standard_normal((1, nh * dv, d))
    Wa = rng.standard_normal((1, nh, d)); Wb = rng.standard_normal((1, nh, d))
    S = oracle.gdn_state(H, A, b, g, Wk, Wv, Wa, Wb, 1e-6, nh, dk, dv)
    sig = lambda z: 1 / (1 + math.exp(-z))
    for h in range(nh):
        M = [[0.0] * dk for _ in range(dv)]
        for t in range(rows):
            x = [sum(A[0, j, i] * H[t, i] for i in range(d)) + b[0, j] for j in range(d)]
            r = math.sqrt(sum(z * z for z in x) / d + 1e-6)
            u = [x[j] / r * g[0, j] for j in range(d)]
            kk = [sum(u[j] * Wk[0, h * dk + c, j] for j in range(d)) for c in range(dk)]
            nk = math.sqrt(sum(z * z for z in kk) + 1e-6)
            kk = [z / nk for z in kk]
            vv = [sum(u[j] * Wv[0, h * dv + c, j] for j in range(d)) for c in range(dv)]
            al = sig(sum(u[j] * Wa[0, h, j] for j in range(d)))
            be = sig(sum(u[j] * Wb[0, h, j] for j in range(d)))
            Mk = [sum(M[i][c] * kk[c] for c in range(dk)) for i in range(dv)]
            M = [[al * (M[i][c] - be * Mk[i] * kk[c]) + be * vv[i] * kk[c] for c in range(dk)]
                 for i in range(dv)]
        np.testing.assert_allclose(S[0, h], np.array(M), rtol=1e-10, atol=1e-12)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_figure4_filled_share():
    """Figure 4: 200 rows, the last 50 exact; constant gates 0.90 and 0.995."""
    gd = _golden("figure4_gate_share.json")
    for case in gd["cases"]:
        share = oracle.filled_weight_share(np.full(gd["rows"], case["gate"]), gd["rows"] - gd["tail"])
        assert abs(share - case["printed_share"]) <= case["printed_tolerance"]
        g, n, t = case["gate"], gd["rows"], gd["tail"]
        assert abs(share - (g ** t - g ** n) / (1 - g ** n)) < 1e-12


def test_speedup_ceiling_printed_values():
    gd = _golden("speedup_ceiling.json")
    for case in gd["cases"]:
        r = oracle.speedup_ceiling(gd["S"], gd["L"], gd["T"], case["N"])
        assert abs(1 / r - case["printed_speedup"]) <= 0.005
        if "printed_r" in case:
            assert abs(r - case["printed_r"]) <= 0.005
