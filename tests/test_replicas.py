"""The replicated (N > 1) measurement path of bench.py, on CPU with gloo.

The fill shards into independent replicas (one prompt per GPU, no data-path
collective); the only cross-rank steps are the barrier and the max over ranks of
the timed region, and the whole-job rate counts every replica's units.
"""
import importlib.util
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        ms = [12.5, 20.0][rank]  # replica 1 is the slowest
        got = b.max_over_ranks(ms, world, torch.device("cpu"))
        rate = b.whole_job_rate(1000.0, world, got)
        # the reference arm runs on rank 0 alone; the other ranks print nothing
        args = type("A", (), {"fit": True})()
        buf = io.StringIO()
        with redirect_stdout(buf):
            b.run_reference(args)
        out[rank] = (got, rate, buf.getvalue())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_time_and_whole_job_rate():
    world = 2
    port = 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        got, rate, text = res[r]
        assert got == 20.0
        assert rate == pytest.approx(1000.0 * 2 / 0.020)
    assert json.loads(res[0][2])["impl"] == "reference"
    assert res[1][2] == ""


def test_single_rank_is_its_own_max():
    b = _bench()
    assert b.max_over_ranks(7.25, 1, torch.device("cpu")) == 7.25
    assert b.whole_job_rate(500.0, 1, 10.0) == pytest.approx(50000.0)
