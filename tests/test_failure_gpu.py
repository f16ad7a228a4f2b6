"""Failure detection on the GPU without a fault: a bounded device wait that nothing
satisfies runs out, records its site in the device error word and returns; the
host reads the code and the context keeps working.
"""
import time

import pytest
import torch

from synthetic import WORKLOADS, fill_inputs
from tests._fill_helpers import new_cache, to_cuda

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from late_layer_kv_gb300 import device_error, ridgefill_fill, wait_selftest  # noqa: E402


@pytest.mark.parametrize("which", [0, 1])
def test_wait_runs_out_and_context_stays_usable(which):
    assert device_error() == 0
    t0 = time.time()
    wait_selftest(which)
    assert device_error() == 20 + which  # synchronises, reads and clears the word
    assert 1.0 < time.time() - t0 < 30.0
    assert device_error() == 0
    shape = WORKLOADS["tiny_d256"]
    d = to_cuda(fill_inputs(shape, seed=1))
    Kc, Vc = new_cache(shape.n_layers, shape.n_kv, shape.N, shape.head_dim)
    ridgefill_fill(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                   head_dim=shape.head_dim, rope_theta=shape.rope_theta, rms_eps=shape.rms_eps)
    assert device_error() == 0
    assert bool(torch.isfinite(Kc[:, :, :shape.rows].float()).all())
