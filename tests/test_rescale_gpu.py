"""GPU parity of ridgefill_rescale (value / key rescale of the filled rows) against
the f64 oracle.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
section 2.3 ("Value rescale") and section 6.6 (the key scale).
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import WORKLOADS, fill_inputs, tail_inputs, to_f64
from tests._fill_helpers import SENTINEL, compare, new_cache, oracle_inputs, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import (  # noqa: E402
    RF_RESCALE_KEYS, RF_RESCALE_VALUES, device_error, ridgefill_fill, ridgefill_rescale)

# The scale is a mean of norm ratios of bf16-rounded projections (one rounding of
# g * x_hat and one of the stored projection, each ~2^-9 per element and
# averaging over the head's elements and the rows): relative error well below 2e-3.
SCALE_RTOL = 2e-3


def _case(name, c, rows, pos0, seed, zero_head=False):
    shape = WORKLOADS[name]
    inp = fill_inputs(shape, seed=seed, rows=1)
    tail = tail_inputs(shape, seed=seed, c=c)
    if zero_head:  # head 1 projects to zero: no usable row, scale 1
        hd = shape.head_dim
        inp["Wv"][:, hd:2 * hd] = 0
        inp["Wk"][:, hd:2 * hd] = 0
    cache_len = pos0 + rows + 16
    g = torch.Generator().manual_seed(seed)
    Kc = torch.full((shape.n_layers, shape.n_kv, cache_len, shape.head_dim), SENTINEL,
                    dtype=torch.bfloat16)
    Vc = Kc.clone()
    Kc[:, :, pos0:pos0 + rows] = torch.randn(shape.n_layers, shape.n_kv, rows, shape.head_dim,
                                             generator=g).bfloat16()
    Vc[:, :, pos0:pos0 + rows] = torch.randn(shape.n_layers, shape.n_kv, rows, shape.head_dim,
                                             generator=g).bfloat16()
    return shape, inp, tail, Kc, Vc


def _run(shape, inp, tail, Kc, Vc, which, rows, pos0):
    d = {k: v.cuda() for k, v in list(inp.items()) + list(tail.items())}
    K, V = Kc.cuda(), Vc.cuda()
    scale = torch.full((shape.n_layers, shape.n_kv), float("nan"), device="cuda")
    ridgefill_rescale(d["H_tail"], d["X_true"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], K, V,
                      which=which, head_dim=shape.head_dim, rms_eps=shape.rms_eps, rows=rows,
                      pos0=pos0, scale=scale)
    torch.cuda.synchronize()
    assert device_error() == 0
    return K.cpu(), V.cpu(), scale.cpu()


def _oracle_scale(shape, inp, tail, which, layers=None):
    o = oracle_inputs(inp)
    W = o["Wv"] if which == RF_RESCALE_VALUES else o["Wk"]
    Ls = range(shape.n_layers) if layers is None else layers
    sel = list(Ls)
    return oracle.kv_rescale(to_f64(tail["H_tail"]), to_f64(tail["X_true"])[sel], o["A"][sel],
                             o["b"][sel], o["g"][sel], W[sel], shape.rms_eps, shape.n_kv,
                             shape.head_dim)


def _check_apply(before, after, scale, rows, pos0):
    want = (before[:, :, pos0:pos0 + rows].float() * scale[:, :, None, None]).bfloat16()
    assert torch.equal(after[:, :, pos0:pos0 + rows], want), "scaled rows differ from bf16(x * s)"
    assert torch.equal(after[:, :, :pos0], before[:, :, :pos0]), "rows before pos0 changed"
    assert torch.equal(after[:, :, pos0 + rows:], before[:, :, pos0 + rows:]), "rows after changed"


@pytest.mark.parametrize("which", [RF_RESCALE_VALUES, RF_RESCALE_KEYS])
@pytest.mark.parametrize("c", [37, 300])
def test_scale_and_apply_small(which, c):
    shape, inp, tail, Kc, Vc = _case("tiny_d256", c=c, rows=200, pos0=5, seed=71)
    K, V, s = _run(shape, inp, tail, Kc, Vc, which, rows=200, pos0=5)
    ref = _oracle_scale(shape, inp, tail, which)
    np.testing.assert_allclose(s.double().numpy(), ref, rtol=SCALE_RTOL)
    assert np.abs(ref - 1.0).max() > 0.02, "test inputs should move the scale away from 1"
    scaled, other = (V, K) if which == RF_RESCALE_VALUES else (K, V)
    _check_apply(Vc if which == RF_RESCALE_VALUES else Kc, scaled, s, 200, 5)
    assert torch.equal(other, Kc if which == RF_RESCALE_VALUES else Vc), "the other cache changed"


def test_single_tail_row_and_zero_head():
    shape, inp, tail, Kc, Vc = _case("tiny_d256", c=1, rows=64, pos0=0, seed=72, zero_head=True)
    K, V, s = _run(shape, inp, tail, Kc, Vc, RF_RESCALE_VALUES, rows=64, pos0=0)
    ref = _oracle_scale(shape, inp, tail, RF_RESCALE_VALUES)
    np.testing.assert_allclose(s.double().numpy(), ref, rtol=SCALE_RTOL)
    assert torch.all(s[:, 1] == 1.0)
    _check_apply(Vc, V, s, 64, 0)


def test_full_size_scales_sampled_layers():
    # Llama-shaped late layers, c = 512 tail rows; the oracle checks three of the 20 layers
    shape, inp, tail, Kc, Vc = _case("llama8b_16k", c=512, rows=4096, pos0=0, seed=73)
    K, V, s = _run(shape, inp, tail, Kc, Vc, RF_RESCALE_VALUES, rows=4096, pos0=0)
    layers = [0, 9, 19]
    ref = _oracle_scale(shape, inp, tail, RF_RESCALE_VALUES, layers=layers)
    np.testing.assert_allclose(s[layers].double().numpy(), ref, rtol=SCALE_RTOL)
    _check_apply(Vc, V, s, 4096, 0)


@pytest.mark.parametrize("which", [RF_RESCALE_VALUES, RF_RESCALE_KEYS])
def test_scales_only_then_fused_fill(which):
    """rows = 0 leaves the caches alone; the scales passed to the fill multiply the
    filled values (keys) of each head, the other half unchanged."""
    shape = WORKLOADS["tiny_d256"]
    inp = fill_inputs(shape, seed=74)
    tail = tail_inputs(shape, seed=74, c=150)
    d = to_cuda(inp)
    t = to_cuda(tail)
    Kc, Vc = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
    scale = torch.full((shape.n_layers, shape.n_kv), float("nan"), device="cuda")
    ridgefill_rescale(t["H_tail"], t["X_true"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                      which=which, head_dim=shape.head_dim, rms_eps=shape.rms_eps, rows=0,
                      scale=scale)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert bool((Kc == SENTINEL).all()) and bool((Vc == SENTINEL).all()), "rows = 0 wrote the cache"
    ref = _oracle_scale(shape, inp, tail, which)
    np.testing.assert_allclose(scale.cpu().double().numpy(), ref, rtol=SCALE_RTOL)
    kw = {"v_scale": scale} if which == RF_RESCALE_VALUES else {"k_scale": scale}
    ridgefill_fill(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                   head_dim=shape.head_dim, rope_theta=shape.rope_theta, rms_eps=shape.rms_eps,
                   **kw)
    torch.cuda.synchronize()
    assert device_error() == 0
    o = oracle_inputs(inp)
    rows = shape.rows
    K, V = oracle.fill_attention(o["H"], np.arange(rows), o["A"], o["b"], o["g"], o["Wk"],
                                 o["Wv"], shape.rms_eps, shape.rope_theta, shape.n_kv,
                                 shape.head_dim)
    if which == RF_RESCALE_VALUES:
        V = V * ref[:, :, None, None]
    else:
        K = K * ref[:, :, None, None]
    gk, gv = to_f64(Kc[:, :, :rows]), to_f64(Vc[:, :, :rows])
    for l in range(shape.n_layers):
        compare(gk[l], K[l], f"K layer {l}")
        compare(gv[l], V[l], f"V layer {l}")
    assert bool((Kc[:, :, rows:] == SENTINEL).all()) and bool((Vc[:, :, rows:] == SENTINEL).all())


def test_unit_scales_are_bitwise_the_plain_fill():
    shape = WORKLOADS["tiny_d256"]
    inp = fill_inputs(shape, seed=75)
    d = to_cuda(inp)
    ones = torch.ones((shape.n_layers, shape.n_kv), device="cuda")
    out = []
    for kw in ({}, {"k_scale": ones, "v_scale": ones}):
        Kc, Vc = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
        ridgefill_fill(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                       head_dim=shape.head_dim, rope_theta=shape.rope_theta,
                       rms_eps=shape.rms_eps, **kw)
        out.append((Kc, Vc))
    torch.cuda.synchronize()
    assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1])
