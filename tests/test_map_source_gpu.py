"""Maps produced on the host one layer at a time (a caller-supplied map source), and the
library's bounded host waits.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill", section 4.2
(maps held in GPU memory or streamed from the host one layer at a time, identical
outputs).  Here the host side is a callback that writes each layer's map into a pinned
staging buffer, as a loader reading from a file or decompressing would.  A source that
fails or stalls, and a copy engine held up behind earlier work, end the call with a status
instead of a hang; nothing on the GPU faults or waits without a bound.
"""
import ctypes
import time

import pytest
import torch

from synthetic import FillShape, fill_inputs
from tests._fill_helpers import SENTINEL, new_cache, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import RidgeFillError, device_error, ridgefill_fill  # noqa: E402
from late_layer_kv_gb300 import ridgefill_quantize_maps  # noqa: E402

SHAPE = FillShape("src", d=512, n_layers=5, n_kv=4, head_dim=128, rope_theta=5e5,
                  rms_eps=1e-6, N=700, T=60)
KW = dict(head_dim=SHAPE.head_dim, rope_theta=SHAPE.rope_theta, rms_eps=SHAPE.rms_eps)


def _inputs(seed):
    inp = fill_inputs(SHAPE, seed=seed)
    return inp, to_cuda(inp)


def _resident(d, A=None, A_scale=None, rpc=0):
    Kc, Vc = new_cache(SHAPE.n_layers, SHAPE.n_kv, SHAPE.N, SHAPE.head_dim)
    ridgefill_fill(d["H"], d["A"] if A is None else A, d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                   rows_per_chunk=rpc, A_scale=A_scale, **KW)
    return Kc, Vc


class LayerSource:
    """Copies layer l of maps held in ordinary (pageable) host memory into the staging
    half; optionally fails or sleeps at one layer.  Records the calls it got."""

    def __init__(self, codes, scales=None, fail_at=-1, sleep_at=-1, sleep_s=0.0):
        self.codes, self.scales = codes.contiguous(), scales
        self.fail_at, self.sleep_at, self.sleep_s = fail_at, sleep_at, sleep_s
        self.calls = []

    def __call__(self, layer, dst, nbytes):
        self.calls.append(layer)
        if layer == self.fail_at:
            return -3
        if layer == self.sleep_at:
            time.sleep(self.sleep_s)
        c = self.codes[layer]
        n = c.numel() * c.element_size()
        ctypes.memmove(dst, c.data_ptr(), n)
        if self.scales is not None:
            s = self.scales[layer].contiguous()
            off = (n + 255) // 256 * 256
            ctypes.memmove(dst + off, s.data_ptr(), s.numel() * s.element_size())
            n = off + s.numel() * s.element_size()
        assert n == nbytes
        return 0


def _sourced(d, src, staging, A_scale=None, rpc=0, wait_ms=0):
    Kc, Vc = new_cache(SHAPE.n_layers, SHAPE.n_kv, SHAPE.N, SHAPE.head_dim)
    ridgefill_fill(d["H"], None, d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc, rows_per_chunk=rpc,
                   A_scale=A_scale, map_source=src, map_staging=staging, host_wait_ms=wait_ms,
                   map_shape=(SHAPE.n_layers, SHAPE.d, SHAPE.d), **KW)
    return Kc, Vc


def _staging(nbytes_per_layer):
    return torch.empty(2 * nbytes_per_layer, dtype=torch.uint8).pin_memory()


def test_sourced_maps_bitwise_equal_resident():
    inp, d = _inputs(41)
    K0, V0 = _resident(d)
    st = _staging(SHAPE.d * SHAPE.d * 2)
    for rpc in (0, 256):  # one chunk, then three: the source is asked once per chunk and layer
        src = LayerSource(inp["A"])
        K1, V1 = _sourced(d, src, st, rpc=rpc)
        torch.cuda.synchronize()
        assert device_error() == 0
        assert torch.equal(K1, K0) and torch.equal(V1, V0), rpc
        assert src.calls == list(range(SHAPE.n_layers)) * (1 if rpc == 0 else 3)


def test_sourced_int8_maps_bitwise_equal_resident():
    inp, d = _inputs(42)
    q, s = ridgefill_quantize_maps(d["A"])
    K0, V0 = _resident(d, A=q, A_scale=s)
    n = SHAPE.d * SHAPE.d
    st = _staging((n + 255) // 256 * 256 + SHAPE.d * (SHAPE.d // 128) * 2)
    src = LayerSource(q.cpu(), s.cpu())
    # a non-NULL A_scale selects int8 maps; its contents are not read with a source
    K1, V1 = _sourced(d, src, st, A_scale=s)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(K1, K0) and torch.equal(V1, V0)


def test_failing_source_returns_its_status_and_leaves_the_context_usable():
    inp, d = _inputs(43)
    st = _staging(SHAPE.d * SHAPE.d * 2)
    src = LayerSource(inp["A"], fail_at=2)
    with pytest.raises(RidgeFillError) as ex:
        _sourced(d, src, st)
    assert ex.value.status == 9 and "layer 2" in str(ex.value)
    assert src.calls == [0, 1, 2]
    torch.cuda.synchronize()
    assert device_error() == 0
    K0, V0 = _resident(d)
    K1, V1 = _sourced(d, LayerSource(inp["A"]), st)
    torch.cuda.synchronize()
    assert torch.equal(K1, K0) and torch.equal(V1, V0)


def test_stalling_source_times_out():
    inp, d = _inputs(44)
    st = _staging(SHAPE.d * SHAPE.d * 2)
    src = LayerSource(inp["A"], sleep_at=1, sleep_s=0.4)
    t0 = time.perf_counter()
    with pytest.raises(RidgeFillError) as ex:
        _sourced(d, src, st, wait_ms=100)
    assert ex.value.status == 6 and "map_source took" in str(ex.value)
    assert time.perf_counter() - t0 < 5.0
    torch.cuda.synchronize()
    assert device_error() == 0


def test_copy_engine_held_up_times_out_on_the_host():
    """The copies of layers 0 and 1 queue behind a bounded spin kernel (about a second) on
    the same stream; the staging half of layer 2 is still waiting to be copied out when the
    50 ms bound runs out, so the call returns RF_ERR_TIMEOUT.  The spin ends by itself, the
    queued work then completes, and the K/V of the chunk were never enqueued."""
    inp, d = _inputs(45)
    st = _staging(SHAPE.d * SHAPE.d * 2)
    Kc, Vc = new_cache(SHAPE.n_layers, SHAPE.n_kv, SHAPE.N, SHAPE.head_dim)
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000_000)
    src = LayerSource(inp["A"])
    with pytest.raises(RidgeFillError) as ex:
        ridgefill_fill(d["H"], None, d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc, map_source=src,
                       map_staging=st, host_wait_ms=50,
                       map_shape=(SHAPE.n_layers, SHAPE.d, SHAPE.d), **KW)
    assert ex.value.status == 6 and "staging" in str(ex.value)
    assert src.calls == [0, 1]
    torch.cuda.synchronize()
    assert device_error() == 0
    assert bool((Kc == SENTINEL).all()) and bool((Vc == SENTINEL).all())
