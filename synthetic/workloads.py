"""Workload shapes and seeded generators.

Every random tensor is drawn block by block: block ``i`` of a tensor with key
``k`` comes from ``numpy.random.PCG64(SeedSequence([*k, i]))``.  The bytes
therefore depend only on the seed and the key, never on thread count, device
or which other tensors were drawn, so the oracle and the GPU path read the
same inputs.

Distributions (the paper replaces real hidden states with these):

* split state ``H`` and calibration ``X``: ``N(0,1) * s_c`` per channel with
  ``s_c ~ LogNormal(0, 1)``, one ``s_c`` vector per workload seed;
* maps ``A_l = I + 0.1 G_l / sqrt(d)``, ``G_l ~ N(0,1)``; biases ``~ N(0,1)``;
* projection weights ``~ N(0, 1/d)``; norm gains ``1 + 0.1 N(0,1)``;
* calibration targets ``Y_l = X (I + 0.1 G_l/sqrt(d)) + b_l + 0.05 N(0,1)``.

bf16 tensors are rounded from float32 with round-to-nearest-even (torch).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from typing import Dict, Optional, Sequence, Tuple

import numpy as np
import torch

_BLOCK = 1 << 22
_THREADS = max(1, min(32, os.cpu_count() or 1))

# tensor ids used in keys (stable; never renumber)
_ID_SCALES, _ID_H, _ID_A, _ID_B, _ID_GAIN, _ID_WK, _ID_WV = 1, 2, 3, 4, 5, 6, 7
_ID_WA, _ID_WB, _ID_X, _ID_YG, _ID_YB, _ID_YN = 8, 9, 10, 11, 12, 13
_ID_TAILH, _ID_TAILX, _ID_TAILS = 14, 15, 16
_ID_EXACT, _ID_XEX, _ID_XEXS = 17, 18, 19


def normal(shape: Sequence[int], key: Tuple[int, ...]) -> np.ndarray:
    """Standard normal float32 array of ``shape``, reproducible from ``key``."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)
    nblk = (n + _BLOCK - 1) // _BLOCK

    def fill(i: int) -> None:
        lo, hi = i * _BLOCK, min(n, (i + 1) * _BLOCK)
        seq = np.random.SeedSequence([int(k) for k in key] + [i])
        np.random.Generator(np.random.PCG64(seq)).standard_normal(
            out=out[lo:hi], dtype=np.float32)

    if nblk <= 1:
        if n:
            fill(0)
    else:
        with ThreadPoolExecutor(min(_THREADS, nblk)) as ex:
            list(ex.map(fill, range(nblk)))
    return out.reshape(tuple(shape))


def channel_scales(d: int, seed: int) -> np.ndarray:
    """Per-channel scales ``s_c = exp(N(0,1))`` (lognormal(0,1)), float32."""
    return np.exp(normal((d,), (seed, _ID_SCALES))).astype(np.float32)


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a (bf16/f32) tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


@dataclass(frozen=True)
class FillShape:
    """Shape of one late-layer fill workload (attention layers).

    ``n_layers`` is the number of late (filled) layers; ``N`` the prompt
    length and ``T`` the exact tail, so rows ``0 .. N-T-1`` are filled.
    """
    name: str
    d: int
    n_layers: int
    n_kv: int
    head_dim: int
    rope_theta: float
    rms_eps: float
    N: int
    T: int
    n_q: int = 0
    total_layers: int = 0
    split: int = 0
    calib_rows: int = 0
    lam: float = 1e-3

    @property
    def rows(self) -> int:
        return self.N - self.T

    @property
    def kv_width(self) -> int:
        return self.n_kv * self.head_dim

    def with_rows(self, N: int, T: int) -> "FillShape":
        return replace(self, N=N, T=T)


@dataclass(frozen=True)
class GdnShape:
    """Hybrid workload: Gated DeltaNet late layers plus attention late layers."""
    name: str
    d: int
    layer_kinds: Tuple[str, ...]      # per late layer: "gdn" or "attn"
    n_heads: int                      # GDN heads
    d_k: int
    d_v: int
    chunk: int
    n_kv: int                         # attention kv heads
    head_dim: int
    rope_theta: float
    rms_eps: float
    N: int
    T: int
    split: int = 0

    @property
    def rows(self) -> int:
        return self.N - self.T

    @property
    def n_gdn(self) -> int:
        return sum(1 for k in self.layer_kinds if k == "gdn")

    @property
    def n_attn(self) -> int:
        return sum(1 for k in self.layer_kinds if k == "attn")

    def attn_shape(self) -> FillShape:
        return FillShape(self.name + "_attn", self.d, self.n_attn, self.n_kv, self.head_dim,
                         self.rope_theta, self.rms_eps, self.N, self.T)


def _hybrid_kinds(total: int, split: int) -> Tuple[str, ...]:
    # every fourth layer (0-indexed 3, 7, 11, ...) is attention, the rest GDN
    return tuple("attn" if (l + 1) % 4 == 0 else "gdn" for l in range(split, total))


WORKLOADS: Dict[str, object] = {}


def _reg(s):
    WORKLOADS[s.name] = s
    return s


# tiny fit + fill: 8 layers, split after layer 2 -> 6 late layers
_reg(FillShape("tiny_d256", d=256, n_layers=6, n_kv=2, head_dim=64, rope_theta=1e4,
               rms_eps=1e-6, N=512, T=64, n_q=4, total_layers=8, split=2,
               calib_rows=4096, lam=1e-3))
# Llama-3.1-8B-shaped fill, maps resident in HBM
_reg(FillShape("llama8b_16k", d=4096, n_layers=20, n_kv=8, head_dim=128, rope_theta=5e5,
               rms_eps=1e-6, N=16384, T=2048, n_q=32, total_layers=32, split=12,
               calib_rows=65536, lam=1e-3))
# 27B-class dense shape, prompt sweep
for _n in (16384, 32768, 65536, 120000):
    _tag = {16384: "16k", 32768: "32k", 65536: "64k", 120000: "120k"}[_n]
    _reg(FillShape(f"dense27b_{_tag}", d=5120, n_layers=43, n_kv=8, head_dim=128,
                   rope_theta=1e6, rms_eps=1e-6, N=_n, T=4096, n_q=64, total_layers=64,
                   split=21))
# host-memory maps: llama8b shapes
for _n, _tag in ((16384, "16k"), (65536, "64k")):
    _reg(FillShape(f"hostmaps_{_tag}", d=4096, n_layers=20, n_kv=8, head_dim=128,
                   rope_theta=5e5, rms_eps=1e-6, N=_n, T=2048, n_q=32, total_layers=32,
                   split=12, calib_rows=65536, lam=1e-3))
# hybrid Gated DeltaNet: 32 layers, split after 12 -> 15 GDN + 5 attention late layers
_reg(GdnShape("hybrid_gdn_32k", d=4096, layer_kinds=_hybrid_kinds(32, 12), n_heads=16,
              d_k=128, d_v=128, chunk=64, n_kv=8, head_dim=128, rope_theta=5e5,
              rms_eps=1e-6, N=32768, T=4096, split=12))


def _maps(n_layers: int, d_out: int, d_in: int, seed: int, layer_ids: Sequence[int]):
    """``A_l = I + 0.1 G_l / sqrt(d)`` as bf16 [L, d_out, d_in]."""
    out = torch.empty((n_layers, d_out, d_in), dtype=torch.bfloat16)
    s = 0.1 / math.sqrt(d_in)
    for i, lid in enumerate(layer_ids):
        g = normal((d_out, d_in), (seed, _ID_A, lid))
        g *= s
        idx = np.arange(min(d_out, d_in))
        g[idx, idx] += 1.0
        out[i] = _bf16(g)
    return out


def _per_layer(n: int, shape, seed: int, tid: int, layer_ids, scale=1.0, shift=0.0):
    arrs = []
    for lid in layer_ids:
        a = normal(shape, (seed, tid, lid))
        if scale != 1.0:
            a *= scale
        if shift != 0.0:
            a += shift
        arrs.append(a)
    return np.stack(arrs) if arrs else np.zeros((0,) + tuple(shape), np.float32)


def _split_state(rows: int, d: int, seed: int, tid: int) -> torch.Tensor:
    s = channel_scales(d, seed)
    h = normal((rows, d), (seed, tid))
    h *= s[None, :]
    return _bf16(h)


def fill_inputs(shape: FillShape, seed: int, layer_ids: Optional[Sequence[int]] = None,
                rows: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Inputs of an attention-layer fill, as CPU tensors.

    Returns ``H`` [rows, d] bf16, ``A`` [L, d, d] bf16 (paper orientation:
    row ``j`` of ``A_l`` produces output channel ``j``), ``b`` [L, d] f32,
    ``g`` [L, d] bf16, ``Wk``/``Wv`` [L, n_kv*hd, d] bf16 (``[out, in]``).
    """
    L, d = shape.n_layers, shape.d
    lids = list(layer_ids) if layer_ids is not None else list(range(L))
    nr = shape.rows if rows is None else rows
    out = {
        "H": _split_state(nr, d, seed, _ID_H),
        "A": _maps(len(lids), d, d, seed, lids),
        "b": torch.from_numpy(_per_layer(L, (d,), seed, _ID_B, lids)),
        "g": _bf16(_per_layer(L, (d,), seed, _ID_GAIN, lids, scale=0.1, shift=1.0)),
        "Wk": _bf16(_per_layer(L, (shape.kv_width, d), seed, _ID_WK, lids,
                               scale=1.0 / math.sqrt(d))),
        "Wv": _bf16(_per_layer(L, (shape.kv_width, d), seed, _ID_WV, lids,
                               scale=1.0 / math.sqrt(d))),
    }
    return out


def tail_inputs(shape: FillShape, seed: int, c: int) -> Dict[str, torch.Tensor]:
    """Rows of the exact tail for the value/key rescale, as CPU tensors.

    ``H_tail`` [c, d] bf16 split states drawn like ``H`` (same per-channel
    scales), and ``X_true`` [L, c, d] bf16 standing in for the true late-layer
    inputs: ``N(0, 1)`` per entry times per-layer, per-channel scales
    ``exp(N(0, 1))`` of their own.
    """
    L, d = shape.n_layers, shape.d
    xt = np.stack([normal((c, d), (seed, _ID_TAILX, l)) *
                   np.exp(normal((d,), (seed, _ID_TAILS, l)))[None, :] for l in range(L)])
    return {"H_tail": _split_state(c, d, seed, _ID_TAILH), "X_true": _bf16(xt.astype(np.float32))}


def exact_rows(rows: int, frac: float, seed: int) -> torch.Tensor:
    """A seeded set of exact prefix rows: about ``frac`` of ``rows``, drawn
    uniformly without replacement, as sorted int32 indices (CPU)."""
    n = int(round(frac * rows))
    pick = np.argsort(normal((rows,), (seed, _ID_EXACT)))[:n]
    return torch.from_numpy(np.sort(pick).astype(np.int32))


def true_inputs(n_layers: int, n: int, d: int, seed: int) -> torch.Tensor:
    """Stand-ins for ``n`` rows' true late-layer inputs, [n_layers, n, d] bf16:
    ``N(0, 1)`` times per-layer, per-channel scales ``exp(N(0, 1))``."""
    x = np.stack([normal((n, d), (seed, _ID_XEX, l)) *
                  np.exp(normal((d,), (seed, _ID_XEXS, l)))[None, :] for l in range(n_layers)])
    return _bf16(x.astype(np.float32))


def gdn_inputs(shape: GdnShape, seed: int, rows: Optional[int] = None,
               gate_scale: float = 1.0) -> Dict[str, torch.Tensor]:
    """Inputs of the hybrid fill.  Late layer ``i`` uses key id ``i`` whatever
    its kind, so the attention and GDN groups are disjoint draws.

    GDN group: ``A``, ``b``, ``g`` as in :func:`fill_inputs`; ``Wk`` [L, H*dk, d],
    ``Wv`` [L, H*dv, d], ``Wa``/``Wb`` [L, H, d], all ``N(0, gate_scale^2/d)``
    for the gates and ``N(0, 1/d)`` otherwise.  Attention group under ``attn_*``.
    """
    d = shape.d
    nr = shape.rows if rows is None else rows
    gl = [i for i, k in enumerate(shape.layer_kinds) if k == "gdn"]
    al = [i for i, k in enumerate(shape.layer_kinds) if k == "attn"]
    sd = 1.0 / math.sqrt(d)
    out = {"H": _split_state(nr, d, seed, _ID_H)}
    for tag, lids in (("", gl), ("attn_", al)):
        n = len(lids)
        out[tag + "A"] = _maps(n, d, d, seed, lids)
        out[tag + "b"] = torch.from_numpy(_per_layer(n, (d,), seed, _ID_B, lids))
        out[tag + "g"] = _bf16(_per_layer(n, (d,), seed, _ID_GAIN, lids, scale=0.1, shift=1.0))
    H, dk, dv = shape.n_heads, shape.d_k, shape.d_v
    out["Wk"] = _bf16(_per_layer(len(gl), (H * dk, d), seed, _ID_WK, gl, scale=sd))
    out["Wv"] = _bf16(_per_layer(len(gl), (H * dv, d), seed, _ID_WV, gl, scale=sd))
    out["Wa"] = _bf16(_per_layer(len(gl), (H, d), seed, _ID_WA, gl, scale=sd * gate_scale))
    out["Wb"] = _bf16(_per_layer(len(gl), (H, d), seed, _ID_WB, gl, scale=sd))
    kw = shape.n_kv * shape.head_dim
    out["attn_Wk"] = _bf16(_per_layer(len(al), (kw, d), seed, _ID_WK, al, scale=sd))
    out["attn_Wv"] = _bf16(_per_layer(len(al), (kw, d), seed, _ID_WV, al, scale=sd))
    return out


def calibration(d: int, n_layers: int, n: int, seed: int, device: str = "cpu",
                layer_ids: Optional[Sequence[int]] = None) -> Dict[str, torch.Tensor]:
    """Calibration pairs ``X`` [n, d] bf16 and ``Y`` [L, n, d] bf16.

    ``Y_l = X (I + 0.1 G_l/sqrt(d)) + b_l + 0.05 N(0,1)`` with ``X`` taken
    after its bf16 rounding; the product is evaluated in float32 on
    ``device`` (data generation only).  Also returns the generating ``M``
    [L, d, d] (row-vector form) and ``bgen`` [L, d] in float32.
    """
    lids = list(layer_ids) if layer_ids is not None else list(range(n_layers))
    s = channel_scales(d, seed)
    x = normal((n, d), (seed, _ID_X))
    x *= s[None, :]
    X = _bf16(x)
    Xd = X.to(device=device, dtype=torch.float32)
    Y = torch.empty((len(lids), n, d), dtype=torch.bfloat16)
    Ms, bs = [], []
    for i, lid in enumerate(lids):
        g = normal((d, d), (seed, _ID_YG, lid))
        g *= 0.1 / math.sqrt(d)
        idx = np.arange(d)
        g[idx, idx] += 1.0
        bg = normal((d,), (seed, _ID_YB, lid))
        nz = normal((n, d), (seed, _ID_YN, lid))
        M = torch.from_numpy(g).to(device)
        y = Xd @ M + torch.from_numpy(bg).to(device)[None, :] + 0.05 * torch.from_numpy(nz).to(device)
        Y[i] = y.to(torch.bfloat16).cpu()
        Ms.append(torch.from_numpy(g))
        bs.append(torch.from_numpy(bg))
    return {"X": X, "Y": Y, "M": torch.stack(Ms), "bgen": torch.stack(bs)}


def calibration_device(d: int, n_layers: int, n: int, seed: int, device) -> Dict[str, torch.Tensor]:
    """Full-size calibration pairs drawn on the device (torch's Philox generator, seeded),
    in the distributions of :func:`calibration`: ``X`` [n, d] bf16 = N(0,1) times
    per-channel LogNormal(0,1) scales, ``Y`` [L, n, d] bf16 = X (I + 0.1 G_l/sqrt(d)) + b_l
    + 0.05 N(0,1).  For sizes whose host generation would take minutes (the full fit
    workload); the bytes depend on the seed and the device's generator, not on numpy."""
    g = torch.Generator(device=device).manual_seed(seed)
    sc = torch.exp(torch.randn(d, generator=g, device=device))
    X = (torch.randn(n, d, generator=g, device=device) * sc).to(torch.bfloat16)
    Y = torch.empty((n_layers, n, d), dtype=torch.bfloat16, device=device)
    Xf = X.float()
    for l in range(n_layers):
        M = torch.eye(d, device=device) + 0.1 * torch.randn(d, d, generator=g, device=device) / d ** 0.5
        bl = torch.randn(d, generator=g, device=device)
        Y[l] = (Xf @ M + bl + 0.05 * torch.randn(n, d, generator=g, device=device)).to(torch.bfloat16)
    return {"X": X, "Y": Y}

