#!/usr/bin/env python
"""Benchmark of the RidgeFill late-layer cache fill on GB300.

One step = one ridgefill_fill call over the whole prefix of one synthetic
prompt: the grouped map GEMM for every late layer and the K/V GEMM that writes
the caches.  The metric is filled token-layers per second ((N - T) * L_late /
step time), also reported as fill-stage ms and as a fraction of the bf16
tensor peak.  With torchrun (N > 1) every rank fills its own prompt (replicas,
no collective on the data path); the timing takes the max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import WORKLOADS, fill_inputs, to_f64  # noqa: E402

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch of the map GEMM from an ncu capture, valid only for the
# kernel source with this digest (otherwise reported as null).
PROFILED_TRAFFIC = {
    "kernel_sha256": None,
    "map_gemm_bytes_per_launch": None,
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def _kernel_digest() -> str:
    h = hashlib.sha256()
    for f in ("fill_gemm.cu", "sm103_ptx.cuh", "rf_internal.h"):
        with open(os.path.join(ROOT, "late_layer_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _flops_per_row_layer(shape) -> float:
    # map d_in*d_out plus the layer's K and V projections, 2 flops per MAC
    return 2.0 * (shape.d * shape.d + shape.d * 2 * shape.kv_width)


def cpu_oracle_rate(shape, inp, sample_rows: int):
    """Filled token-layers/s of the f64 oracle on a seeded row sample."""
    import oracle
    o = {k: to_f64(v) for k, v in inp.items()}
    idx = np.sort(np.random.default_rng(0).choice(shape.rows, size=sample_rows, replace=False))
    t0 = time.perf_counter()
    oracle.fill_attention(o["H"][idx], idx, o["A"], o["b"], o["g"], o["Wk"], o["Wv"],
                          shape.rms_eps, shape.rope_theta, shape.n_kv, shape.head_dim)
    dt = time.perf_counter() - t0
    return sample_rows * shape.n_layers / dt, dt


def _cores():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v):
            return int(os.environ[v])
    return os.cpu_count() or 1


def run_reference(args, shape):
    world, rank, _ = _dist()
    if rank != 0:
        return
    inp = fill_inputs(shape, seed=1001)
    sample = args.ref_rows
    rates, times = [], []
    for i in range(args.warmup + args.steps):
        r, dt = cpu_oracle_rate(shape, inp, sample)
        if i >= args.warmup:
            rates.append(r)
            times.append(dt)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "token-layers/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * float(np.mean(times)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(shape),
        "cpu_baseline": {"value": value, "unit": "token-layers/s", "cores": _cores(),
                         "kind": "oracle",
                         "sample": f"{sample} seeded random prefix rows x all {shape.n_layers} "
                                   f"late layers per step"},
        "e2e": {"value": value, "unit": "token-layers/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "filled token-layers/s (fill-stage ms and % of GB300 bf16 tensor peak alongside)"


def _config(shape):
    return {"workload": shape.name, "d": shape.d, "late_layers": shape.n_layers, "N": shape.N,
            "T": shape.T, "filled_rows": shape.rows, "kv_heads": shape.n_kv,
            "head_dim": shape.head_dim, "maps": "hbm",
            "l2": "inputs larger than L2 (maps %d MiB, split state %d MiB)" % (
                shape.n_layers * shape.d * shape.d * 2 >> 20, shape.rows * shape.d * 2 >> 20)}



def _e2e(shape, inp, d, Kc, Vc, ws, stream, steps, world, dev, token_layers):
    """The same metric through the public call with host buffers: each step copies the
    prompt's split state H from pinned host memory and reads two cache rows per layer back."""
    from late_layer_kv_gb300 import ridgefill_fill
    L, rows = shape.n_layers, shape.rows
    H_host = inp["H"].pin_memory()
    out_host = torch.empty((L, shape.n_kv, 2, shape.head_dim), dtype=torch.bfloat16).pin_memory()
    H_dev = torch.empty_like(d["H"])

    def one():
        H_dev.copy_(H_host, non_blocking=True)
        ridgefill_fill(H_dev, d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                       head_dim=shape.head_dim, rope_theta=shape.rope_theta,
                       rms_eps=shape.rms_eps, workspace=ws, stream=stream)
        out_host.copy_(Kc[:, :, rows - 2:rows], non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / steps
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    return {"value": token_layers * world / (e2e_ms / 1000.0), "unit": "token-layers/s",
            "ms_per_step": e2e_ms, "h2d_bytes_per_step": int(H_host.numel() * 2),
            "d2h_bytes_per_step": int(out_host.numel() * 2)}

def run_ours(args, shape):
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from late_layer_kv_gb300 import device_error, ridgefill_fill
    from late_layer_kv_gb300 import ridgefill as rb

    inp = fill_inputs(shape, seed=1001 + rank)
    d = {k: v.to(dev) for k, v in inp.items()}
    L, rows = shape.n_layers, shape.rows
    Kc = torch.zeros((L, shape.n_kv, shape.N, shape.head_dim), dtype=torch.bfloat16, device=dev)
    Vc = torch.zeros_like(Kc)
    ws_args = rb.fill_args(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                           head_dim=shape.head_dim, rope_theta=shape.rope_theta,
                           rms_eps=shape.rms_eps)
    ws = torch.empty(rb.fill_workspace_size(ws_args), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in sum(ev, []):
        e.record(stream)  # torch creates the CUDA event on first record

    def step(i=None):
        ridgefill_fill(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], Kc, Vc,
                       head_dim=shape.head_dim, rope_theta=shape.rope_theta,
                       rms_eps=shape.rms_eps, workspace=ws, stream=stream,
                       stage_events=None if i is None else ev[i])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert device_error(stream) == 0

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    assert device_error(stream) == 0
    ms = t0.elapsed_time(t1)
    map_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ev]))
    kv_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in ev]))
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    ms_step = ms / steps
    token_layers = rows * L
    value = token_layers * world / (ms_step / 1000.0)

    # end to end through the public call with host buffers: pinned H in, a cache row out
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(shape, inp, d, Kc, Vc, ws, stream, steps, world, dev, token_layers)

    peaks, src = _peaks()
    # a timed region of a few seconds or more runs under the power cap: compare with the
    # sustained cuBLAS figure; shorter regions with the burst figure
    sustained = ms >= 2000.0
    peak_key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = float(peaks[peak_key])
    map_flops = 2.0 * rows * L * shape.d * shape.d
    achieved = map_flops / (map_ms / 1000.0) / 1e12
    total_flops = rows * L * _flops_per_row_layer(shape)
    pct = 100.0 * total_flops / (ms_step / 1000.0) / 1e12 / peak
    traffic = None
    if PROFILED_TRAFFIC["kernel_sha256"] == _kernel_digest():
        traffic = PROFILED_TRAFFIC["map_gemm_bytes_per_launch"]

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        r, dt = cpu_oracle_rate(shape, inp, args.cpu_rows)
        cpu = {"value": r, "unit": "token-layers/s", "cores": _cores(), "kind": "oracle",
               "sample": f"{args.cpu_rows} seeded random prefix rows x all {L} late layers "
                         f"({dt:.1f} s of f64 numpy work)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "token-layers/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": _config(shape),
            "fill_stage_ms": ms_step, "map_gemm_ms": map_ms, "kv_gemm_ms": kv_ms,
            "pct_bf16_peak": pct,
            "roofline": {"bound": "tensor", "kernel": "map GEMM (rf_gemm_kernel, map mode)",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": f"{src} {peak_key}",
                         "timed_region_ms": ms},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 2 * steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama8b_16k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=4096)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--rows", type=int, default=0, help="override the filled rows (profiling)")
    ap.add_argument("--layers", type=int, default=0, help="override the late layers (profiling)")
    args = ap.parse_args()
    shape = WORKLOADS[args.workload]
    if args.rows or args.layers:
        from dataclasses import replace
        rows = args.rows or shape.rows
        L = args.layers or shape.n_layers
        shape = replace(shape, name=f"{shape.name}_rows{rows}_L{L}", N=rows + shape.T,
                        n_layers=L)
    if args.impl == "reference":
        run_reference(args, shape)
    else:
        run_ours(args, shape)


if __name__ == "__main__":
    main()
