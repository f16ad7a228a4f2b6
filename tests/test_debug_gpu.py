"""The debug build of the library (every plain global store of the kernels checked
against its buffer, a guard band after every workspace region, filled before and checked
after each call) on the paths the release tests cover: no check fires, and the results
are bitwise those of the release library.

This stands in for a memory checker, which is not available on the GPUs these tests run
on.  A check that fired would be reported through the device error word as RF_ERR_BOUNDS.
"""
import numpy as np
import pytest
import torch

from synthetic import FillShape, GdnShape, exact_rows, fill_inputs, gdn_inputs, true_inputs
from tests._fill_helpers import new_cache, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import (FitSums, debug_library, device_error,  # noqa: E402
                                 ridgefill_fill, ridgefill_fill_gdn, ridgefill_fit_accumulate,
                                 ridgefill_fit_solve, ridgefill_quantize_maps, ridgefill_rescale)


def _both(run):
    """run() under the release library, then under the debug one; both device error words
    must stay clear."""
    out_r = run()
    torch.cuda.synchronize()
    assert device_error() == 0
    with debug_library():
        out_d = run()
        torch.cuda.synchronize()
        assert device_error() == 0, "a debug check fired"
    return out_r, out_d


def _equal(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_fill_paths_debug_equals_release():
    shape = FillShape("dbg", d=512, n_layers=3, n_kv=4, head_dim=128, rope_theta=5e5,
                      rms_eps=1e-6, N=1000, T=77)
    inp = fill_inputs(shape, seed=51)
    d = to_cuda(inp)
    kw = dict(head_dim=128, rope_theta=5e5, rms_eps=1e-6)
    keep = np.ones(shape.rows, bool)
    keep[exact_rows(shape.rows, 0.3, seed=51).numpy()] = False
    ridx = torch.from_numpy(np.nonzero(keep)[0].astype(np.int32)).cuda()
    A_host = inp["A"].pin_memory()
    H_host = inp["H"].pin_memory()
    q, s = ridgefill_quantize_maps(d["A"])
    cases = [dict(), dict(rows_per_chunk=256), dict(row_idx=ridx), dict(A=A_host),
             dict(H=H_host), dict(A=q, A_scale=s), dict(A=q, A_scale=s, q8_group_layers=-1)]
    for case in cases:
        def run(case=case):
            Kc, Vc = new_cache(3, 4, shape.N, 128)
            c = dict(case)
            H = c.pop("H", d["H"])
            A = c.pop("A", d["A"])
            ridgefill_fill(H, A, d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc, **kw, **c)
            return Kc, Vc
        r, g = _both(run)
        _equal(r, g)


def test_gdn_debug_equals_release():
    shape = GdnShape("dbg_gdn", d=256, layer_kinds=("gdn",) * 2, n_heads=8, d_k=128, d_v=128,
                     chunk=64, n_kv=2, head_dim=128, rope_theta=1e4, rms_eps=1e-6, N=500, T=0)
    inp = gdn_inputs(shape, seed=52)
    d = {k: v.cuda() for k, v in inp.items()}
    ex = exact_rows(shape.rows, 0.2, seed=52).cuda()
    X = true_inputs(2, ex.numel(), 256, seed=52).cuda()
    dM = 1e-3 * torch.randn((2, 8, 128, 128), generator=torch.Generator().manual_seed(1)).cuda()
    for case in (dict(), dict(rows_per_chunk=128),
                 dict(exact_idx=ex, X_exact=X, delta_M=dM)):
        def run(case=case):
            S = torch.empty((2, 8, 128, 128), device="cuda")
            rho = torch.empty((2, 8), device="cuda")
            extra = dict(case)
            if "delta_M" in extra:
                extra["rho"] = rho
            ridgefill_fill_gdn(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], d["Wa"], d["Wb"],
                               S, n_heads=8, rms_eps=1e-6, **extra)
            return S, rho if "delta_M" in case else S
        r, g = _both(run)
        _equal(r, g)


def test_fit_and_rescale_debug_equal_release():
    from synthetic import calibration, tail_inputs
    L, dm, n = 3, 256, 1000
    cal = calibration(dm, L, n, seed=53)
    X, Y = cal["X"].cuda(), cal["Y"].cuda()

    def fit():
        sums = FitSums(L, dm, dm)
        ridgefill_fit_accumulate(sums, X, Y)
        A = torch.empty((L, dm, dm), dtype=torch.bfloat16, device="cuda")
        b = torch.empty((L, dm), dtype=torch.float32, device="cuda")
        ridgefill_fit_solve(sums, 1e-3, A_out=A, b_out=b)
        return A, b, sums.G, sums.C
    r, g = _both(fit)
    _equal(r, g)

    shape = FillShape("dbg_rs", d=256, n_layers=2, n_kv=2, head_dim=128, rope_theta=1e4,
                      rms_eps=1e-6, N=600, T=100)
    inp = to_cuda(fill_inputs(shape, seed=54))
    t = to_cuda(tail_inputs(shape, seed=54, c=37))

    def rescale():
        Kc, Vc = new_cache(2, 2, shape.N, 128)
        ridgefill_fill(inp["H"], inp["A"], inp["b"], inp["g"], inp["Wk"], inp["Wv"], Kc, Vc,
                       head_dim=128, rope_theta=1e4, rms_eps=1e-6)
        sc = torch.empty((2, 2), device="cuda")
        ridgefill_rescale(t["H_tail"], t["X_true"], inp["A"], inp["b"], inp["g"], inp["Wk"],
                          inp["Wv"], Kc, Vc, which=1, head_dim=128, rms_eps=1e-6,
                          rows=shape.rows, scale=sc)
        return Kc, Vc, sc
    r, g = _both(rescale)
    _equal(r, g)
