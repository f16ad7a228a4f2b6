"""Shared helpers for the GPU parity tests of the fill."""
import numpy as np
import torch

from synthetic import to_f64

# Tolerances for bf16-in / f32-accumulate K, V and states against the f64 oracle:
# relative Frobenius error and max element error relative to the reference RMS.
REL_FRO = 5e-3
MAX_REL_RMS = 3e-2


def compare(got: np.ndarray, ref: np.ndarray, what: str, rel_fro=REL_FRO, max_rel_rms=MAX_REL_RMS):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = got - ref
    rf = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    rms = np.sqrt(np.mean(ref * ref))
    mx = np.abs(err).max() / max(rms, 1e-300)
    assert rf <= rel_fro, f"{what}: relative Frobenius error {rf:.3e} > {rel_fro}"
    assert mx <= max_rel_rms, f"{what}: max error {mx:.3e} x rms > {max_rel_rms}"
    return rf, mx


def to_cuda(inp: dict, device="cuda") -> dict:
    return {k: v.to(device) for k, v in inp.items()}


SENTINEL = -12288.0  # exactly representable in bf16 (-3 * 2^12)


def new_cache(L, n_kv, cache_len, hd, device="cuda"):
    Kc = torch.full((L, n_kv, cache_len, hd), SENTINEL, dtype=torch.bfloat16, device=device)
    Vc = torch.full((L, n_kv, cache_len, hd), SENTINEL, dtype=torch.bfloat16, device=device)
    return Kc, Vc


def oracle_inputs(inp: dict) -> dict:
    return {k: to_f64(v) for k, v in inp.items()}
