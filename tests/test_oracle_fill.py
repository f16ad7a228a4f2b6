"""Pins of the oracle's attention-layer fill.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
sections 2.1 and 2.2 (map, the layer's own norm and projections, rotary
embedding on keys) and Table 3 (identity fill).
"""
import cmath
import math

import numpy as np

import oracle


def _brute_fill_row(h, A, b, g, Wk, Wv, pos, eps, theta, hd):
    """One row, one layer, pure Python loops."""
    d_out, d_in = len(A), len(A[0])
    x = [sum(A[j][i] * h[i] for i in range(d_in)) + b[j] for j in range(d_out)]
    ms = sum(v * v for v in x) / d_out
    u = [x[j] / math.sqrt(ms + eps) * g[j] for j in range(d_out)]
    k = [sum(u[j] * Wk[c][j] for j in range(d_out)) for c in range(len(Wk))]
    v = [sum(u[j] * Wv[c][j] for j in range(d_out)) for c in range(len(Wv))]
    out_k = list(k)
    for h0 in range(0, len(k), hd):
        for i in range(hd // 2):
            ang = pos * theta ** (-2.0 * i / hd)
            a, c = k[h0 + i], k[h0 + i + hd // 2]
            out_k[h0 + i] = a * math.cos(ang) - c * math.sin(ang)
            out_k[h0 + i + hd // 2] = c * math.cos(ang) + a * math.sin(ang)
    return out_k, v


def test_brute_force_tiny():
    rng = np.random.default_rng(0)
    d, n_kv, hd, rows, L = 8, 2, 4, 3, 2
    H = rng.standard_normal((rows, d))
    A = rng.standard_normal((L, d, d))
    b = rng.standard_normal((L, d))
    g = 1 + 0.1 * rng.standard_normal((L, d))
    Wk = rng.standard_normal((L, n_kv * hd, d))
    Wv = rng.standard_normal((L, n_kv * hd, d))
    pos = np.array([0, 7, 123456])
    K, V = oracle.fill_attention(H, pos, A, b, g, Wk, Wv, 1e-6, 1e4, n_kv, hd)
    for l in range(L):
        for r in range(rows):
            bk, bv = _brute_fill_row(H[r].tolist(), A[l].tolist(), b[l].tolist(), g[l].tolist(),
                                     Wk[l].tolist(), Wv[l].tolist(), int(pos[r]), 1e-6, 1e4, hd)
            np.testing.assert_allclose(K[l, :, r, :].reshape(-1), bk, rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(V[l, :, r, :].reshape(-1), bv, rtol=1e-10, atol=1e-10)


def test_identity_fill_is_layer_kv_of_split_state():
    """A = I, b = 0 (the identity fill of Table 3) writes the layer's own K/V of H."""
    rng = np.random.default_rng(1)
    d, n_kv, hd, rows = 16, 2, 8, 5
    H = rng.standard_normal((rows, d))
    g = 1 + 0.1 * rng.standard_normal((1, d))
    Wk = rng.standard_normal((1, n_kv * hd, d))
    Wv = rng.standard_normal((1, n_kv * hd, d))
    pos = np.arange(rows) + 3
    K, V = oracle.fill_attention(H, pos, np.eye(d)[None], np.zeros((1, d)), g, Wk, Wv,
                                 1e-6, 1e4, n_kv, hd)
    K2, V2 = oracle.late_layer_kv(H, g[0], Wk[0], Wv[0], pos, 1e-6, 1e4, n_kv, hd)
    np.testing.assert_array_equal(K[0], K2)
    np.testing.assert_array_equal(V[0], V2)


def test_rope_position_zero_is_identity():
    k = np.random.default_rng(2).standard_normal((3, 4, 128))
    np.testing.assert_array_equal(oracle.rope_rotate_half(k, np.zeros(4), 5e5), k)


def test_rope_matches_complex_rotation():
    """Rotate-half RoPE = multiplying (k_i + i k_{i+hd/2}) by exp(i pos theta^{-2i/hd})."""
    rng = np.random.default_rng(3)
    hd, theta = 16, 1e6
    k = rng.standard_normal((5, hd))
    pos = np.array([0, 1, 17, 4096, 119999])
    out = oracle.rope_rotate_half(k, pos, theta)
    for r in range(5):
        for i in range(hd // 2):
            z = complex(k[r, i], k[r, i + hd // 2]) * cmath.exp(1j * pos[r] * theta ** (-2 * i / hd))
            assert abs(out[r, i] - z.real) < 1e-12 and abs(out[r, i + hd // 2] - z.imag) < 1e-12


def test_rope_preserves_pair_norms_and_is_relative():
    rng = np.random.default_rng(4)
    hd = 64
    q = rng.standard_normal((1, hd))
    k = rng.standard_normal((1, hd))
    for m, n in ((3, 11), (1000, 70000)):
        km = oracle.rope_rotate_half(k, np.array([n]), 1e4)
        pn = np.hypot(km[0, :hd // 2], km[0, hd // 2:])
        np.testing.assert_allclose(pn, np.hypot(k[0, :hd // 2], k[0, hd // 2:]), rtol=1e-12)
        d1 = oracle.rope_rotate_half(q, np.array([m]), 1e4) @ km.T
        d2 = (oracle.rope_rotate_half(q, np.array([m + 500]), 1e4)
              @ oracle.rope_rotate_half(k, np.array([n + 500]), 1e4).T)
        np.testing.assert_allclose(d1, d2, rtol=1e-9)


def test_rmsnorm_scale_invariance():
    """With b = 0, scaling the split state leaves K and V unchanged (up to eps)."""
    rng = np.random.default_rng(5)
    d, n_kv, hd, rows = 32, 1, 16, 4
    H = rng.standard_normal((rows, d))
    A = rng.standard_normal((1, d, d))
    g = 1 + 0.1 * rng.standard_normal((1, d))
    Wk = rng.standard_normal((1, n_kv * hd, d))
    Wv = rng.standard_normal((1, n_kv * hd, d))
    pos = np.arange(rows)
    z = np.zeros((1, d))
    K1, V1 = oracle.fill_attention(H, pos, A, z, g, Wk, Wv, 0.0, 1e4, n_kv, hd)
    K2, V2 = oracle.fill_attention(9.0 * H, pos, A, z, g, Wk, Wv, 0.0, 1e4, n_kv, hd)
    np.testing.assert_allclose(K1, K2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(V1, V2, rtol=1e-12, atol=1e-12)


def test_rmsnorm_unit_rms():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((7, 40)) * 30
    u = oracle.rms_norm(x, np.ones(40), 0.0)
    np.testing.assert_allclose(np.sqrt((u * u).mean(-1)), 1.0, rtol=1e-12)
