"""Plain, slow, float64 CPU oracle of the RidgeFill late-layer fill and fit.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library.

Source of every formula: "RidgeFill: Training-Free Late-Layer Cache Fill for
Faster Prefill" (arXiv 2611.09709), section and equation named on each
function.  All inputs are widened to float64; nothing is rounded in between.
Matrix products, the Cholesky factor and triangular solves are library
primitives (numpy / scipy); nothing is blocked, fused or reordered.

Notation.  The paper writes column vectors, ``x_hat = A x_S + b`` with ``A``
of shape ``d_out x d_in``.  Arrays here hold one row per token, so a batch of
predictions is ``H @ A.T + b``; ``A`` keeps the paper's orientation.

Readings where the paper is silent (each applied below):

* R1 ridge centring: ``X`` and ``Y`` in the closed form are mean-centred and
  the offset ``b`` is unpenalised (section 2.2: means subtracted, offset makes
  the map right on average).
* R2 penalty trace: ``alpha = lambda * tr(X^T X) / d_in`` uses the centred X,
  the matrix that enters the solve.
* R3 layer norm: RMSNorm with a plain gain, ``x / sqrt(mean(x^2) + eps) * g``.
* R4 rotary embedding: rotate-half pairs ``(i, i + hd/2)``, frequency
  ``theta^(-2i/hd)``, position = absolute prompt row; keys only.
* R5 Gated DeltaNet: gates read the normed input ``u`` like ``k`` and ``v``,
  ``alpha = sigmoid(u . w_a)``, ``beta = sigmoid(u . w_b)``, no short
  convolution; ``k`` is L2-normalised with ``k / sqrt(sum k^2 + 1e-6)``; state
  ``S`` is ``d_v x d_k`` and starts at zero unless given.
* R6 rows: every prefix row is filled; the tail is not touched.
* R16 value/key rescale: "the ratio of the exact value norm to the predicted
  one, averaged over the c rows" is the mean of the per-row ratios.
* R19 exact prefix rows (section 2.4): an exact row's late-layer input is its
  true input, given; in an attention layer the fill does not write its row, in
  a GDN layer it enters the state in prompt order with its true input.
* R20 rho (section 2.3, terminal-state correction): the weight of row t in the
  state at the end of the prefix is the product of the gates of the rows after
  it; rho is taken per layer and head (the gates are per head; Delta M is per
  value head), over the prefix rows only.
* R18 int8 maps: symmetric absmax groups of 128 consecutive weights of a row,
  scale ``s = bf16(absmax / 127)``, code ``q = rint(a / s)`` (ties to even,
  clamped to [-127, 127]); an all-zero group has ``s = 0``, ``q = 0``.  The
  two divisions that decide ``s`` and ``q`` are IEEE float32 operations, the
  precision of the kernel that makes the codes; everything after is float64.

Parity status: every function below is pinned by a test in ``tests/`` that
does not re-evaluate its own formula (closed forms, exact rational
arithmetic, library routines for the same textbook problem, invariants, the
paper's printed numbers).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import scipy.linalg


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Fit  (section 2.2, "The ridge map", "Fitting", "The penalty")
# --------------------------------------------------------------------------

def ridge_fit(X, Y, lam: float):
    """Closed-form ridge map per late layer, section 2.2.

    ``X`` [n, d_in] split states, ``Y`` [L, n, d_out] layer inputs.  Both are
    centred by their means (R1); ``alpha = lam * tr(X^T X) / d_in`` (R2);
    ``A_l = Y_l^T X (X^T X + alpha I)^{-1}`` and ``b_l = mu_l - A_l mu_S``.

    Returns ``A`` [L, d_out, d_in], ``b`` [L, d_out], ``alpha``.
    """
    X = _f64(X)
    Y = _f64(Y)
    n, d_in = X.shape
    mu_S = X.mean(axis=0)
    Xc = X - mu_S
    G = Xc.T @ Xc
    alpha = lam * np.trace(G) / d_in
    chol = scipy.linalg.cho_factor(G + alpha * np.eye(d_in), lower=True)
    L = Y.shape[0]
    A = np.empty((L, Y.shape[2], d_in))
    b = np.empty((L, Y.shape[2]))
    for l in range(L):
        mu_l = Y[l].mean(axis=0)
        Yc = Y[l] - mu_l
        # (X^T X + alpha I) is symmetric, so A_l^T = (X^T X + alpha I)^{-1} X^T Y_l
        A[l] = scipy.linalg.cho_solve(chol, Xc.T @ Yc).T
        b[l] = mu_l - A[l] @ mu_S
    return A, b, alpha


def fit_sums(X, Y):
    """Running sums of one capture pass, section 2.2 "Fitting".

    Returns ``(n, sx, sy, G, C)``: row count, ``sum x`` [d_in], ``sum y_l``
    [L, d_out], ``X^T X`` [d_in, d_in] and ``X^T Y_l`` as [d_in, L*d_out]
    (column block ``l`` holds layer ``l``).  Uncentred; additive over rows.
    """
    X = _f64(X)
    Y = _f64(Y)
    L = Y.shape[0]
    G = X.T @ X
    C = np.concatenate([X.T @ Y[l] for l in range(L)], axis=1)
    return X.shape[0], X.sum(axis=0), Y.sum(axis=1), G, C


def ridge_solve_from_sums(n, sx, sy, G, C, lam: float):
    """The same solve as :func:`ridge_fit`, from the running sums.

    Centring of sums: ``X~^T X~ = G - n mu_S mu_S^T`` and
    ``X~^T Y~_l = C_l - n mu_S mu_l^T``.
    """
    sx, sy, G, C = _f64(sx), _f64(sy), _f64(G), _f64(C)
    d_in = G.shape[0]
    L, d_out = sy.shape
    mu_S = sx / n
    mu = sy / n
    Gc = G - n * np.outer(mu_S, mu_S)
    alpha = lam * np.trace(Gc) / d_in
    chol = scipy.linalg.cho_factor(Gc + alpha * np.eye(d_in), lower=True)
    A = np.empty((L, d_out, d_in))
    b = np.empty((L, d_out))
    for l in range(L):
        Cl = C[:, l * d_out:(l + 1) * d_out] - n * np.outer(mu_S, mu[l])
        A[l] = scipy.linalg.cho_solve(chol, Cl).T
        b[l] = mu[l] - A[l] @ mu_S
    return A, b, alpha


# --------------------------------------------------------------------------
# Fill, attention layers  (section 2.1, 2.2 "At inference ...")
# --------------------------------------------------------------------------

def map_apply(H, A_l, b_l):
    """``x_hat = A_l x_S + b_l`` for every row of ``H`` [rows, d_in] (section 2.2)."""
    return _f64(H) @ _f64(A_l).T + _f64(b_l)


def rms_norm(x, g, eps: float):
    """The layer's own normalisation applied to a predicted input (R3)."""
    x = _f64(x)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * _f64(g)


def rope_rotate_half(k, pos, theta: float):
    """Rotary embedding of keys ``k`` [..., rows, hd] at positions ``pos`` [rows] (R4)."""
    k = _f64(k)
    hd = k.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / hd)
    ang = _f64(pos)[:, None] * inv_freq[None, :]
    c, s = np.cos(ang), np.sin(ang)
    k1, k2 = k[..., :half], k[..., half:]
    return np.concatenate([k1 * c - k2 * s, k2 * c + k1 * s], axis=-1)


def late_layer_kv(x_hat, g, Wk, Wv, pos, eps: float, theta: float, n_kv: int, hd: int):
    """What a late attention layer writes for predicted inputs ``x_hat`` [rows, d].

    Section 2.1/2.2: the layer's own norm, its key and value projections
    (``Wk``, ``Wv`` as [n_kv*hd, d]) and the rotary embedding on keys.
    Returns ``K``, ``V`` as [n_kv, rows, hd].
    """
    u = rms_norm(x_hat, g, eps)
    rows = u.shape[0]
    k = (u @ _f64(Wk).T).reshape(rows, n_kv, hd).transpose(1, 0, 2)
    v = (u @ _f64(Wv).T).reshape(rows, n_kv, hd).transpose(1, 0, 2)
    return rope_rotate_half(k, pos, theta), v


def fill_attention(H, pos, A, b, g, Wk, Wv, eps: float, theta: float, n_kv: int, hd: int,
                   layers: Optional[Sequence[int]] = None):
    """The late-layer cache fill for the given prefix rows (sections 2.1-2.2).

    ``H`` [rows, d_in] split states of the rows, ``pos`` [rows] their absolute
    positions, ``A`` [L, d_out, d_in], ``b`` [L, d_out], ``g`` [L, d_out],
    ``Wk``/``Wv`` [L, n_kv*hd, d_out].  Returns ``K``, ``V`` as
    [len(layers), n_kv, rows, hd].
    """
    Ls = range(np.shape(A)[0]) if layers is None else layers
    Ks, Vs = [], []
    for l in Ls:
        xh = map_apply(H, A[l], b[l])
        k, v = late_layer_kv(xh, g[l], Wk[l], Wv[l], pos, eps, theta, n_kv, hd)
        Ks.append(k)
        Vs.append(v)
    return np.stack(Ks), np.stack(Vs)


def kv_rescale(H_tail, X_true, A, b, g, W, eps: float, n_kv: int, hd: int):
    """Per-layer, per-kv-head scale of the value (or key) rescale, section 2.3
    "Value rescale" (and the key scale of section 6.6).

    The first ``c`` tail rows go through the layer's norm and projection ``W``
    ([L, n_kv*hd, d_out]: W_v for values, W_k for keys) twice: from their true
    late-layer inputs ``X_true`` [L, c, d_out] and from the map's prediction
    ``A h + b`` of their split states ``H_tail`` [c, d_in].  The scale of a head
    is the mean over the rows of ||exact|| / ||predicted|| (R16: the per-row
    ratio averaged; rows whose predicted norm is 0 are left out, and a head
    with no such row keeps scale 1).  The rotary embedding preserves key norms,
    so it does not enter.  Returns [L, n_kv].
    """
    L = np.shape(A)[0]
    out = np.ones((L, n_kv))
    for l in range(L):
        W_l = _f64(W[l])
        pred = rms_norm(map_apply(H_tail, A[l], b[l]), g[l], eps) @ W_l.T
        true = rms_norm(X_true[l], g[l], eps) @ W_l.T
        for h in range(n_kv):
            cols = slice(h * hd, (h + 1) * hd)
            n_pred = np.sqrt(np.sum(pred[:, cols] ** 2, axis=1))
            n_true = np.sqrt(np.sum(true[:, cols] ** 2, axis=1))
            ok = n_pred > 0
            if ok.any():
                out[l, h] = np.mean(n_true[ok] / n_pred[ok])
    return out


# --------------------------------------------------------------------------
# Fill, Gated DeltaNet layers  (section 2.3)
# --------------------------------------------------------------------------

def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def gdn_projections(x_hat, g, Wk, Wv, Wa, Wb, eps: float, n_heads: int, dk: int, dv: int,
                    l2_eps: float = 1e-6):
    """Per-row ``k`` [rows, H, dk] (L2-normalised), ``v`` [rows, H, dv] and gates
    ``alpha``, ``beta`` [rows, H] of a GDN layer, from its normed input (R5)."""
    u = rms_norm(x_hat, g, eps)
    rows = u.shape[0]
    k = (u @ _f64(Wk).T).reshape(rows, n_heads, dk)
    k = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + l2_eps)
    v = (u @ _f64(Wv).T).reshape(rows, n_heads, dv)
    alpha = _sigmoid(u @ _f64(Wa).T)
    beta = _sigmoid(u @ _f64(Wb).T)
    return k, v, alpha, beta


def gdn_recurrence(k, v, alpha, beta, S0=None):
    """Gated delta rule over rows in order (section 2.3; R5).

    ``S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T`` for every
    head.  ``k`` [rows, H, dk], ``v`` [rows, H, dv], ``alpha``/``beta`` [rows, H];
    ``S`` is [H, dv, dk].  ``S (I - beta k k^T)`` is evaluated as
    ``S - beta (S k) k^T``, the same product written out.
    """
    k, v, alpha, beta = _f64(k), _f64(v), _f64(alpha), _f64(beta)
    rows, nh, dk = k.shape
    dv = v.shape[2]
    S = np.zeros((nh, dv, dk)) if S0 is None else _f64(S0).copy()
    for t in range(rows):
        kt, vt = k[t], v[t]
        a = alpha[t][:, None, None]
        bt = beta[t][:, None, None]
        Sk = np.einsum("hvk,hk->hv", S, kt)
        S = a * (S - bt * Sk[:, :, None] * kt[:, None, :]) + bt * vt[:, :, None] * kt[:, None, :]
    return S


def layer_inputs(H, A_l, b_l, exact_idx=None, X_exact_l=None):
    """Every prefix row's input to one late layer (sections 2.2 and 2.4, R19):
    the map's prediction ``A h + b``, except that the exact rows ``exact_idx``
    take their true inputs ``X_exact_l`` [len(exact_idx), d_out]."""
    x = map_apply(H, A_l, b_l)
    if exact_idx is not None and len(exact_idx) > 0:
        x[np.asarray(exact_idx)] = _f64(X_exact_l)
    return x


def gdn_state(H, A, b, g, Wk, Wv, Wa, Wb, eps: float, n_heads: int, dk: int, dv: int,
              S0=None, layers: Optional[Sequence[int]] = None,
              heads: Optional[Sequence[int]] = None, l2_eps: float = 1e-6,
              exact_idx=None, X_exact=None):
    """End-of-fill recurrent state of GDN late layers (sections 2.1, 2.3).

    Every prefix row, in order, updates the state from its input: the map's
    prediction, or for the exact rows ``exact_idx`` their true inputs
    ``X_exact`` [L, len(exact_idx), d_out] (section 2.4, R19).
    Returns [len(layers), len(heads), dv, dk].
    """
    Ls = range(np.shape(A)[0]) if layers is None else layers
    hs = list(range(n_heads)) if heads is None else list(heads)
    out = []
    for l in Ls:
        xh = layer_inputs(H, A[l], b[l], exact_idx, None if X_exact is None else X_exact[l])
        k, v, a, bt = gdn_projections(xh, g[l], Wk[l], Wv[l], Wa[l], Wb[l], eps,
                                      n_heads, dk, dv, l2_eps)
        s0 = None if S0 is None else _f64(S0)[l][hs]
        out.append(gdn_recurrence(k[:, hs], v[:, hs], a[:, hs], bt[:, hs], s0))
    return np.stack(out)


# --------------------------------------------------------------------------
# Host-side arithmetic (section 2.5, section 2.3 / Figure 4)
# --------------------------------------------------------------------------

def speedup_ceiling(S: int, L: int, T: int, N: int):
    """Share of exact prefill compute that remains, ``r = (S(N-T) + L T)/(L N)``,
    section 2.5; the speedup is at most ``1/r``."""
    return (S * (N - T) + L * T) / (L * N)


def filled_share(alpha, filled):
    """rho of section 2.3 (terminal-state correction, R20): the filled rows'
    total weight over all rows' total weight, where a row's weight in the state
    at the end of the rows is the product of the gates after it.

    ``alpha`` [rows] gates of one head, ``filled`` [rows] bool.  The suffix
    products are a reversed cumulative product (a library primitive).
    """
    a = _f64(alpha)
    f = np.asarray(filled, dtype=bool)
    # w[t] = prod(a[t+1:]): reverse cumulative product, shifted by one
    after = np.concatenate([np.cumprod(a[::-1])[::-1][1:], [1.0]])
    return after[f].sum() / after.sum()


def gdn_rho(H, A, b, g, Wa, eps: float, n_heads: int, exact_idx=None, X_exact=None,
            layers: Optional[Sequence[int]] = None):
    """rho [len(layers), n_heads] of GDN late layers at the end of the prefix:
    per head, ``filled_share`` of the gates the layer computes from every
    prefix row's input (R19, R20)."""
    Ls = range(np.shape(A)[0]) if layers is None else layers
    rows = np.shape(H)[0]
    filled = np.ones(rows, dtype=bool)
    if exact_idx is not None:
        filled[np.asarray(exact_idx, dtype=np.int64)] = False
    out = []
    for l in Ls:
        x = layer_inputs(H, A[l], b[l], exact_idx, None if X_exact is None else X_exact[l])
        alpha = _sigmoid(rms_norm(x, g[l], eps) @ _f64(Wa[l]).T)  # [rows, H] (R5)
        out.append([filled_share(alpha[:, h], filled) for h in range(n_heads)])
    return np.asarray(out)


def terminal_correction(S, rho, delta_M):
    """The state after the terminal-state correction of section 2.3,
    ``S + rho Delta M``, once per layer and head (``S``, ``delta_M``
    [L, H, dv, dk]; ``rho`` [L, H])."""
    return _f64(S) + _f64(rho)[:, :, None, None] * _f64(delta_M)


def filled_weight_share(alpha, n_filled: int):
    """Share of a GDN state that comes from the first ``n_filled`` rows.

    Section 2.3 (terminal-state correction) and Figure 4: a row's weight in
    the final state is the product of the gates after it.  ``alpha`` [rows].
    """
    a = _f64(alpha)
    rows = a.shape[0]
    w = np.empty(rows)
    for t in range(rows):
        w[t] = np.prod(a[t + 1:])
    return w[:n_filled].sum() / w.sum()


# --------------------------------------------------------------------------
# int8 maps  (section 2.2 "Size and cost"; section 4.2 map format)
# --------------------------------------------------------------------------

Q8_GROUP = 128  # weights of a row that share one scale


def _to_bf16(x):
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def quantize_map(A):
    """int8 codes and bf16 scales of maps ``A`` [..., d_out, d_in] (R18).

    Section 2.2 ("Size and cost") and section 4.2 store the maps as int8 with
    one scale per 128 weights of each row.  Returns ``q`` [..., d_out, d_in]
    int8 and ``s`` [..., d_out, d_in / 128] (bf16 values held in float32).
    """
    a = np.asarray(A, dtype=np.float32)
    d_in = a.shape[-1]
    assert d_in % Q8_GROUP == 0
    g = a.reshape(a.shape[:-1] + (d_in // Q8_GROUP, Q8_GROUP))
    amax = np.abs(g).max(axis=-1)
    s = _to_bf16(amax / np.float32(127.0))
    safe = np.where(s > 0, s, np.float32(1.0))
    q = np.rint(g / safe[..., None])
    q = np.where(s[..., None] > 0, np.clip(q, -127, 127), 0)
    return q.reshape(a.shape).astype(np.int8), s


def dequantize_map(q, s):
    """The weights ``q * s`` the int8 maps stand for, float64 [..., d_out, d_in]."""
    qq = np.asarray(q, dtype=np.float64)
    d_in = qq.shape[-1]
    g = qq.reshape(qq.shape[:-1] + (d_in // Q8_GROUP, Q8_GROUP))
    return (g * _f64(s)[..., None]).reshape(qq.shape)
