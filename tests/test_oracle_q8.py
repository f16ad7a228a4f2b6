"""Pins of the oracle's int8 map format (quantize_map / dequantize_map).

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
section 2.2 ("Size and cost": int8 with one scale per 128 weights of each
row; 1.2 GiB for the 27B's 48 maps, 0.60 GiB for Flash-Next's 24) and
section 4.2.
"""
import json
import os

import numpy as np

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "int8_map_sizes.json")


def _bf16_values(rng, n):
    """n random positive floats that bf16 holds exactly (8 significant bits)."""
    mant = rng.integers(128, 256, size=n)
    exp = rng.integers(-12, 2, size=n)
    return (mant / 128.0) * 2.0 ** exp


def test_printed_storage_sizes():
    """One-byte codes in groups of 128 with a 2-byte scale give the printed totals
    to the printed digits.  bf16 maps (2.34 / 1.17 GiB) or groups of 32, llama.cpp's
    Q8_0 block (Flash-Next: 0.62 GiB), would not; the printed digits do not tell a
    2-byte scale from a 4-byte one, the text names bf16."""
    with open(GOLD) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        # the oracle's own output shapes for one map row block, scaled to the full map
        q, s = oracle.quantize_map(np.ones((8, c["d_in"]), np.float32))
        per_row = q.shape[-1] * 1 + s.shape[-1] * 2  # int8 codes, bf16 scales
        total = per_row * c["d_out"] * c["maps"] / 2 ** 30
        assert abs(total - c["printed_gib"]) <= c["printed_tolerance"], (c["model"], total)
        assert s.shape[-1] * oracle.Q8_GROUP == c["d_in"]


def test_exact_multiples_round_trip():
    rng = np.random.default_rng(0)
    rows, d = 6, 512
    s0 = _bf16_values(rng, rows * d // 128).reshape(rows, d // 128)
    k = rng.integers(-127, 128, size=(rows, d))
    k.reshape(rows, d // 128, 128)[:, :, 5] = 127 * rng.choice([-1, 1], size=(rows, d // 128))
    A = (k.reshape(rows, d // 128, 128) * s0[..., None]).reshape(rows, d)
    assert np.array_equal(A.astype(np.float32).astype(np.float64), A)
    q, s = oracle.quantize_map(A)
    assert np.array_equal(s.astype(np.float64), s0)
    assert np.array_equal(q.astype(np.int64), k)
    assert np.array_equal(oracle.dequantize_map(q, s), A)


def test_zero_group_and_bounds():
    rng = np.random.default_rng(1)
    A = rng.standard_normal((3, 4, 384)).astype(np.float32) * np.exp(rng.standard_normal((3, 4, 1)))
    A[1, 2, 128:256] = 0.0
    q, s = oracle.quantize_map(A)
    assert q.dtype == np.int8 and q.shape == A.shape and s.shape == (3, 4, 3)
    assert s[1, 2, 1] == 0 and not q[1, 2, 128:256].any()
    g = q.reshape(3, 4, 3, 128).astype(np.int64)
    nz = s > 0
    assert np.all(np.abs(g).max(axis=-1)[nz] == 127)
    assert np.all(np.abs(g) <= 127)
    err = np.abs(oracle.dequantize_map(q, s) - A.astype(np.float64))
    half = 0.5 * np.repeat(s.astype(np.float64), 128, axis=-1)
    assert np.all(err <= half * (1 + 1e-6))
    # the scale is the group's absmax / 127 to bf16 precision
    amax = np.abs(A.reshape(3, 4, 3, 128)).max(axis=-1).astype(np.float64)
    ratio = s.astype(np.float64)[nz] * 127 / amax[nz]
    assert np.all(np.abs(ratio - 1) <= 2.0 ** -8)


def test_codes_are_nearest_integers_in_f64():
    """Away from exact ties, the f32 decision equals the nearest integer of the
    exact f64 quotient."""
    rng = np.random.default_rng(2)
    A = (rng.standard_normal((16, 1024)) * 0.05).astype(np.float32)
    q, s = oracle.quantize_map(A)
    quot = A.astype(np.float64).reshape(16, 8, 128) / s.astype(np.float64)[..., None]
    frac = np.abs(quot - np.floor(quot) - 0.5)
    ref = np.clip(np.rint(quot), -127, 127)
    ok = frac > 1e-5
    assert np.array_equal(q.reshape(16, 8, 128)[ok].astype(np.float64), ref[ok])
    assert ok.mean() > 0.999
