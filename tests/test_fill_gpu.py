"""GPU parity of ridgefill_fill (attention late layers) against the f64 oracle.

Paper: "RidgeFill: Training-Free Late-Layer Cache Fill for Faster Prefill",
sections 2.1-2.2; section 4.2 (resident and streamed maps give identical
outputs); Table 3 (identity fill).
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic import WORKLOADS, FillShape, fill_inputs, to_f64
from tests._fill_helpers import SENTINEL, compare, new_cache, oracle_inputs, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import device_error, ridgefill_fill  # noqa: E402


def _run(shape: FillShape, inp, pos0=0, cache_len=None, rows_per_chunk=0, host_maps=False,
         gain=True):
    d = to_cuda(inp)
    A = inp["A"].pin_memory() if host_maps else d["A"]
    cache_len = cache_len or (pos0 + shape.rows + shape.T)
    Kc, Vc = new_cache(shape.n_layers, shape.n_kv, cache_len, shape.head_dim)
    ridgefill_fill(d["H"], A, d["b"], d["g"] if gain else None, d["Wk"], d["Wv"], Kc, Vc,
                   head_dim=shape.head_dim, rope_theta=shape.rope_theta, rms_eps=shape.rms_eps,
                   pos0=pos0, rows_per_chunk=rows_per_chunk)
    torch.cuda.synchronize()
    assert device_error() == 0
    return Kc, Vc


def _oracle(shape, inp, rows_idx, pos0=0, layers=None, gain=True):
    o = oracle_inputs(inp)
    g = o["g"] if gain else np.ones_like(o["g"])
    return oracle.fill_attention(o["H"][rows_idx], pos0 + np.asarray(rows_idx), o["A"], o["b"], g,
                                 o["Wk"], o["Wv"], shape.rms_eps, shape.rope_theta, shape.n_kv,
                                 shape.head_dim, layers=layers)


def _check_all(shape, inp, Kc, Vc, pos0=0, gain=True):
    rows = shape.rows
    K, V = _oracle(shape, inp, np.arange(rows), pos0, gain=gain)
    gk = to_f64(Kc[:, :, pos0:pos0 + rows])
    gv = to_f64(Vc[:, :, pos0:pos0 + rows])
    for l in range(shape.n_layers):
        compare(gk[l], K[l], f"K layer {l}")
        compare(gv[l], V[l], f"V layer {l}")
    # nothing outside [pos0, pos0 + rows) is written
    for C in (Kc, Vc):
        outside = torch.cat([C[:, :, :pos0].reshape(-1), C[:, :, pos0 + rows:].reshape(-1)])
        assert bool((outside == SENTINEL).all()), "fill wrote outside the prefix rows"


def test_tiny_full_parity():
    shape = WORKLOADS["tiny_d256"]
    inp = fill_inputs(shape, seed=1000)
    Kc, Vc = _run(shape, inp)
    _check_all(shape, inp, Kc, Vc)


def test_ragged_chunks_offset_positions():
    shape = FillShape("mid", d=512, n_layers=3, n_kv=4, head_dim=128, rope_theta=5e5,
                      rms_eps=1e-6, N=1000 + 77, T=77)
    inp = fill_inputs(shape, seed=7)
    Kc, Vc = _run(shape, inp, pos0=4099, cache_len=4099 + 1000 + 130, rows_per_chunk=256)
    _check_all(shape, inp, Kc, Vc, pos0=4099)


def test_no_gain_and_rows_below_one_tile():
    shape = FillShape("small", d=256, n_layers=2, n_kv=2, head_dim=128, rope_theta=1e4,
                      rms_eps=1e-5, N=37 + 5, T=5)
    inp = fill_inputs(shape, seed=8)
    Kc, Vc = _run(shape, inp, gain=False)
    _check_all(shape, inp, Kc, Vc, gain=False)


def test_empty_prefix_writes_nothing():
    """No prefix rows (N = T): the call succeeds and leaves the whole cache untouched."""
    shape = FillShape("empty", d=256, n_layers=2, n_kv=2, head_dim=128, rope_theta=1e4,
                      rms_eps=1e-6, N=64, T=64)
    inp = fill_inputs(shape, seed=10)
    assert inp["H"].shape[0] == 0
    Kc, Vc = _run(shape, inp, pos0=5, cache_len=64)
    for C in (Kc, Vc):
        assert bool((C == SENTINEL).all())


def test_chunked_equals_unchunked_bitwise():
    shape = FillShape("mid", d=512, n_layers=2, n_kv=2, head_dim=128, rope_theta=5e5,
                      rms_eps=1e-6, N=700, T=0)
    inp = fill_inputs(shape, seed=9)
    K1, V1 = _run(shape, inp)
    K2, V2 = _run(shape, inp, rows_per_chunk=128)
    assert torch.equal(K1, K2) and torch.equal(V1, V2)


def test_host_maps_bitwise_equal_resident():
    """Streaming maps from host memory gives identical caches (section 4.2)."""
    shape = FillShape("mid", d=512, n_layers=5, n_kv=4, head_dim=128, rope_theta=5e5,
                      rms_eps=1e-6, N=640, T=100)
    inp = fill_inputs(shape, seed=10)
    K1, V1 = _run(shape, inp)
    K2, V2 = _run(shape, inp, host_maps=True)
    K3, V3 = _run(shape, inp, host_maps=True, rows_per_chunk=256)
    assert torch.equal(K1, K2) and torch.equal(V1, V2)
    assert torch.equal(K1, K3) and torch.equal(V1, V3)


def test_identity_fill_matches_layer_kv_of_split_state():
    """A = I, b = 0 (identity fill) writes the layer's K/V computed from H itself."""
    shape = FillShape("id", d=256, n_layers=2, n_kv=2, head_dim=64, rope_theta=1e4,
                      rms_eps=1e-6, N=300, T=44)
    inp = fill_inputs(shape, seed=11)
    inp["A"] = torch.eye(256, dtype=torch.bfloat16).expand(2, 256, 256).contiguous()
    inp["b"] = torch.zeros(2, 256)
    Kc, Vc = _run(shape, inp)
    o = oracle_inputs(inp)
    pos = np.arange(shape.rows)
    for l in range(2):
        K, V = oracle.late_layer_kv(o["H"], o["g"][l], o["Wk"][l], o["Wv"][l], pos, shape.rms_eps,
                                    shape.rope_theta, shape.n_kv, shape.head_dim)
        compare(to_f64(Kc[l, :, :shape.rows]), K, "identity K")
        compare(to_f64(Vc[l, :, :shape.rows]), V, "identity V")


def test_bad_arguments_are_rejected():
    """Invalid calls return a status and enqueue nothing (checked at the C ABI)."""
    import ctypes
    from late_layer_kv_gb300 import RidgeFillError, load
    from late_layer_kv_gb300 import ridgefill as rb
    shape = FillShape("bad", d=256, n_layers=1, n_kv=2, head_dim=64, rope_theta=1e4,
                      rms_eps=1e-6, N=10, T=0)
    d = to_cuda(fill_inputs(shape, seed=1))
    Kc, Vc = new_cache(1, 2, 5, 64)  # cache too short for 10 rows
    with pytest.raises(RidgeFillError):
        ridgefill_fill(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc, head_dim=64,
                       rope_theta=1e4, rms_eps=1e-6)
    assert bool((Kc == SENTINEL).all())
    lib = load()
    Kc, Vc = new_cache(1, 2, 16, 64)
    a = rb.fill_args(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc, head_dim=64,
                     rope_theta=1e4, rms_eps=1e-6)
    s = torch.cuda.current_stream().cuda_stream
    host_map = d["A"].cpu()  # pageable, not pinned
    a.maps_on_host = 1
    a.A = host_map.data_ptr()
    ws = torch.empty(rb.fill_workspace_size(a), dtype=torch.uint8, device="cuda")
    assert lib.ridgefill_fill(ctypes.byref(a), ws.data_ptr(), ws.numel(), s) == 4
    a.maps_on_host = 0
    a.A = d["A"].data_ptr()
    a.Kc = Kc.data_ptr() + 2  # misaligned
    assert lib.ridgefill_fill(ctypes.byref(a), ws.data_ptr(), ws.numel(), s) == 3
    a.Kc = Kc.data_ptr()
    assert lib.ridgefill_fill(ctypes.byref(a), ws.data_ptr(), 16, s) == 8  # workspace too small
    torch.cuda.synchronize()
    assert bool((Kc == SENTINEL).all()) and device_error() == 0


@pytest.mark.parametrize("name", ["llama8b_16k"])
def test_full_size_sampled_rows(name):
    """Full-size fill in the benchmark's launch configuration, checked on sampled rows
    (first, last, tile and chunk boundaries, and random rows) of every layer."""
    shape = WORKLOADS[name]
    inp = fill_inputs(shape, seed=1001)
    Kc, Vc = _run(shape, inp)
    rows = shape.rows
    rng = np.random.default_rng(0)
    idx = sorted(set([0, 1, 127, 128, rows // 2, rows - 129, rows - 128, rows - 1]
                     + rng.integers(0, rows, 40).tolist()))
    K, V = _oracle(shape, inp, idx)
    gk = to_f64(Kc[:, :, idx])
    gv = to_f64(Vc[:, :, idx])
    for l in range(shape.n_layers):
        compare(gk[l], K[l], f"K layer {l}")
        compare(gv[l], V[l], f"V layer {l}")
    tail = Kc[:, :, rows:]
    assert bool((tail == SENTINEL).all()) and bool((Vc[:, :, rows:] == SENTINEL).all())


@pytest.mark.parametrize("name", ["hostmaps_16k", "hostmaps_64k"])
def test_full_size_host_maps_sampled_rows(name):
    """The host-map workloads at full size (section 4.2: the 20 maps of 4096 x 4096 stay in
    pinned host memory and are copied one layer at a time while the previous layer's GEMM
    runs), launched as the benchmark launches them: the caches equal those of the same
    fill from device-resident maps bit for bit, and match the oracle on sampled rows
    (first, last, tile and 4096-row group boundaries, 40 random rows) of every layer; the
    tail stays untouched."""
    shape = WORKLOADS[name]
    inp = fill_inputs(shape, seed=1001)
    Kh, Vh = _run(shape, inp, host_maps=True)
    Kd, Vd = _run(shape, inp)
    assert torch.equal(Kh, Kd) and torch.equal(Vh, Vd)
    del Kd, Vd
    rows = shape.rows
    rng = np.random.default_rng(1)
    idx = sorted(set([0, 1, 127, 128, 4095, 4096, rows // 2, rows - 129, rows - 128, rows - 1]
                     + rng.integers(0, rows, 40).tolist()))
    K, V = _oracle(shape, inp, idx)
    gk = to_f64(Kh[:, :, idx])
    gv = to_f64(Vh[:, :, idx])
    for l in range(shape.n_layers):
        compare(gk[l], K[l], f"K layer {l}")
        compare(gv[l], V[l], f"V layer {l}")
    for C in (Kh, Vh):
        assert bool((C[:, :, rows:] == SENTINEL).all()), "fill wrote into the tail rows"


def test_host_split_state_bitwise_equal_device():
    """H in pinned host memory: the library copies it in row groups overlapped with the
    map GEMM; the caches are bitwise those of a device-resident H (several 4096-row
    groups, chunked rows, and host maps as well)."""
    shape = FillShape("hostH", d=512, n_layers=3, n_kv=4, head_dim=128, rope_theta=5e5,
                      rms_eps=1e-6, N=9000 + 100, T=100)
    inp = fill_inputs(shape, seed=12)
    d = to_cuda(inp)
    H_host = inp["H"].pin_memory()
    out = []
    for H, A, rpc in ((d["H"], d["A"], 0), (H_host, d["A"], 0), (H_host, d["A"], 4096),
                      (H_host, inp["A"].pin_memory(), 0)):
        Kc, Vc = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
        ridgefill_fill(H, A, d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc, head_dim=shape.head_dim,
                       rope_theta=shape.rope_theta, rms_eps=shape.rms_eps, rows_per_chunk=rpc)
        out.append((Kc, Vc))
    torch.cuda.synchronize()
    assert device_error() == 0
    K0, V0 = out[0]
    for K, V in out[1:]:
        assert torch.equal(K, K0) and torch.equal(V, V0)


def test_full_size_dense27b_120k_chunked():
    """The 27B-class shape at its longest prompt (d = 5120, 43 late layers, theta = 1e6,
    115,904 prefix rows, positions up to 115,903), launched as the benchmark launches it:
    16,384-row chunks.  Each cache tensor holds 43 * 8 * 120,000 * 128 elements, more
    than 2^31, so the later layers are written at element offsets past 2^31.  Checked on
    every layer at rows 0, 1, the last prefix row, both sides of every chunk boundary and
    40 seeded random rows; the tail rows stay untouched."""
    shape = WORKLOADS["dense27b_120k"]
    rpc = 16384
    inp = fill_inputs(shape, seed=1002)
    Kc, Vc = _run(shape, inp, rows_per_chunk=rpc)
    rows = shape.rows
    assert Kc.numel() > 2 ** 31
    rng = np.random.default_rng(3)
    bounds = [c * rpc + e for c in range(1, -(-rows // rpc)) for e in (-1, 0)]
    idx = sorted(set([0, 1, rows - 1] + bounds + rng.integers(0, rows, 40).tolist()))
    gk = to_f64(Kc[:, :, idx])
    gv = to_f64(Vc[:, :, idx])
    Hs = to_f64(inp["H"][idx])
    for l in range(shape.n_layers):
        K, V = oracle.fill_attention(Hs, np.asarray(idx), to_f64(inp["A"][l:l + 1]),
                                     to_f64(inp["b"][l:l + 1]), to_f64(inp["g"][l:l + 1]),
                                     to_f64(inp["Wk"][l:l + 1]), to_f64(inp["Wv"][l:l + 1]),
                                     shape.rms_eps, shape.rope_theta, shape.n_kv,
                                     shape.head_dim)
        compare(gk[l], K[0], f"K layer {l}")
        compare(gv[l], V[0], f"V layer {l}")
    for C in (Kc, Vc):
        assert bool((C[:, :, rows:] == SENTINEL).all()), "fill wrote into the tail rows"
