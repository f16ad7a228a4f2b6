#!/usr/bin/env python
"""Benchmark of the RidgeFill late-layer fill on GB300.

One step = one pass of the fill over the whole prefix of one synthetic prompt
(N - T filled rows through every late layer).  The metric is filled
token-layers per second: (N - T) * L_late / step time.  Alongside it the line
reports the fill-stage ms, the share of the bf16 tensor peak, per-kernel stage
times (CUDA events recorded by the library between its launches on the
launching stream), the roofline of the dominant kernel, an end-to-end figure
through the public call with host buffers, and the CPU oracle's rate.

Workloads (``--workload``):
  llama8b_16k (default)           attention fill, maps in HBM
  dense27b_{16k,32k,64k,120k}      27B-class dense shape, rows processed in chunks
  hostmaps_{16k,64k}               maps in pinned host memory, streamed per layer
  hybrid_gdn_32k                   15 Gated DeltaNet + 5 attention late layers
With torchrun (N > 1) every rank fills its own prompt (replicas, no collective
on the data path); the timing takes the max over ranks.
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
from dataclasses import replace

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import (WORKLOADS, FillShape, GdnShape, calibration_device,  # noqa: E402
                       exact_rows, fill_inputs, gdn_inputs, tail_inputs, to_f64, true_inputs)

METRIC = "filled token-layers/s (fill-stage ms and % of GB300 bf16 tensor peak alongside)"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}

# DRAM bytes per launch of the dominant kernel from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum, one pass, full size), keyed by the bench line's workload and valid
# only while the library sources that define that kernel hash to kernel_sha256 (otherwise
# reported as null).  The map GEMM's figure comes from a capture of the default fill, the
# Gram accumulate's from a capture of the full fit.
# The fit depends only on d, the number of maps and the calibration rows, which the Llama-8B
# fill workloads share (4096, 20, 65,536): one capture serves all of their fits.
_FIT_LLAMA8B = {"sources": "fit",
                "kernel_sha256": "9b89e6533986f9df6cb73884b54521314b2e6a844b321568addfc22fbedc6876",
                "bytes_per_launch": 85647740160 + 2792289024}
PROFILED_TRAFFIC = {
    "llama8b_16k": {"sources": "fill",
                    "kernel_sha256": "259339cf000223d74faccc3fe2a396ba9465fa5247a05d574d759b2453f90dcb",
                    "bytes_per_launch": 2978276403 + 2344075468},
    "llama8b_16k_fit": _FIT_LLAMA8B,
    "hostmaps_16k_fit": _FIT_LLAMA8B,
    "hostmaps_64k_fit": _FIT_LLAMA8B,
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return PEAKS_FALLBACK, "fallback"


# Sources that define each profiled kernel and its launch: the recorded traffic stays valid
# while these are unchanged.
_SOURCES = {
    "fill": ("abi_common.cu", "abi_common.h", "fill.cu", "fill_gemm.cu", "rf_internal.h",
             "sm103_ptx.cuh"),
    "fit": ("abi_common.cu", "abi_common.h", "fit.cu", "fill_gemm.cu", "rf_internal.h",
            "sm103_ptx.cuh"),
}


def _kernel_digest(which: str = "fill") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "late_layer_kv_gb300", "csrc")
    for f in _SOURCES[which]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines, self.thread = index, None, [], None

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
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's ``x`` (timed regions end when the slowest replica
    does); ``x`` itself with one rank."""
    if world <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units all replicas processed per second over the slowest replica's time."""
    return units_per_rank * world / (ms / 1000.0)


def _cores():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v):
            return int(os.environ[v])
    return os.cpu_count() or 1


def _events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


# ----------------------------------------------------------------------------- workloads

class AttnWorkload:
    """Attention late layers (ridgefill_fill); maps in HBM or in pinned host memory."""

    def __init__(self, shape: FillShape, host_maps=False, rows_per_chunk=0, rescale_rows=0,
                 int8_maps=False, exact_frac=0.0, q8_group=0):
        self.shape, self.host_maps, self.rpc = shape, host_maps, rows_per_chunk
        self.c = rescale_rows
        self.q8 = int8_maps
        self.q8_group = q8_group
        self.exact_frac = exact_frac
        if self.c and host_maps:
            raise ValueError("the rescale needs the maps resident in device memory")
        s = shape
        # with exact prefix rows (section 2.4) only the other rows are filled
        self.n_fill = s.rows - int(round(exact_frac * s.rows))
        self.token_layers = self.n_fill * s.n_layers
        self.stage_names = ["map_gemm", "kv_gemm"]
        self.stage_work = {  # algorithmic FLOP of the first chunk's launches
            "map_gemm": 2.0 * self._chunk_rows() * s.n_layers * s.d * s.d,
            "kv_gemm": 2.0 * self._chunk_rows() * s.n_layers * s.d * 2 * s.kv_width,
        }
        self.stage_bound = {"map_gemm": "tensor", "kv_gemm": "tensor"}
        self.total_flops = 2.0 * self.n_fill * s.n_layers * (s.d * s.d + s.d * 2 * s.kv_width)
        if self.c:
            # value rescale before the fill: the c tail rows' map GEMM and one value
            # projection of the 2c stacked predicted and true rows; the fill applies
            # the per-head scales as it writes the values
            self.stage_names.append("value_rescale")
            self.stage_work["value_rescale"] = 2.0 * self.c * s.n_layers * (
                s.d * s.d + 2 * s.d * s.kv_width)
            self.stage_bound["value_rescale"] = "tensor"
            self.total_flops += self.stage_work["value_rescale"]

    def _chunk_rows(self):
        return min(self.rpc, self.n_fill) if self.rpc else self.n_fill

    def launches_per_step(self):
        chunks = -(-self.n_fill // self._chunk_rows())
        # map GEMM (one per layer with host maps), RoPE table, K/V GEMM
        per_chunk = (self.shape.n_layers + 2) if self.host_maps else 3
        per_chunk += 1 if self.exact_frac else 0  # the row gather
        # rescale: map GEMM, true-input norm, value GEMM, ratio
        return chunks * per_chunk + (4 if self.c else 0)

    def setup(self, dev, seed, inp=None):
        from late_layer_kv_gb300 import ridgefill as rb
        s = self.shape
        self.inp = fill_inputs(s, seed=seed) if inp is None else inp
        self.d = {k: v.to(dev) for k, v in self.inp.items()}
        self.A_scale = None
        if self.q8:  # int8 maps with one bf16 scale per 128 weights, made on the device
            from late_layer_kv_gb300 import ridgefill_quantize_maps
            q, sc = ridgefill_quantize_maps(self.d["A"])
            torch.cuda.synchronize()
            self.d["A"], self.A_scale = q, sc
            if self.host_maps:
                self.A_scale = sc.cpu().pin_memory()
        self.A = self.d["A"].cpu().pin_memory() if self.host_maps else self.d["A"]
        self.Kc = torch.zeros((s.n_layers, s.n_kv, s.N, s.head_dim), dtype=torch.bfloat16,
                              device=dev)
        self.Vc = torch.zeros_like(self.Kc)
        a = rb.fill_args(self.d["H"], self.A, self.d["b"], self.d["g"], self.d["Wk"],
                         self.d["Wv"], self.Kc, self.Vc, head_dim=s.head_dim,
                         rope_theta=s.rope_theta, rms_eps=s.rms_eps, rows_per_chunk=self.rpc,
                         A_scale=self.A_scale, q8_group_layers=self.q8_group)
        self.row_idx = None
        if self.exact_frac:
            keep = np.ones(s.rows, bool)
            keep[exact_rows(s.rows, self.exact_frac, seed=seed).numpy()] = False
            self.row_idx = torch.from_numpy(np.nonzero(keep)[0].astype(np.int32)).to(dev)
            assert self.row_idx.numel() == self.n_fill
            a = rb.fill_args(self.d["H"], self.A, self.d["b"], self.d["g"], self.d["Wk"],
                             self.d["Wv"], self.Kc, self.Vc, head_dim=s.head_dim,
                             rope_theta=s.rope_theta, rms_eps=s.rms_eps, rows_per_chunk=self.rpc,
                             A_scale=self.A_scale, row_idx=self.row_idx,
                             q8_group_layers=self.q8_group)
        self.ws = torch.empty(rb.fill_workspace_size(a), dtype=torch.uint8, device=dev)
        self.H_dev = self.d["H"]
        if self.c:
            t = {k: v.to(dev) for k, v in tail_inputs(s, seed=seed, c=self.c).items()}
            self.tail = t
            self.scale = torch.empty((s.n_layers, s.n_kv), dtype=torch.float32, device=dev)
            ra = rb.rescale_args(t["H_tail"], t["X_true"], self.A, self.d["b"], self.d["g"],
                                 self.d["Wk"], self.d["Wv"], self.Kc, self.Vc,
                                 which=rb.RF_RESCALE_VALUES, head_dim=s.head_dim,
                                 rms_eps=s.rms_eps, rows=0, scale=self.scale,
                                 A_scale=self.A_scale)
            self.rws = torch.empty(max(1, rb.load().ridgefill_rescale_workspace_size(
                ctypes_byref(ra))), dtype=torch.uint8, device=dev)

    def n_events(self):
        return 3 + (2 * self.shape.n_layers if self.host_maps else 0) + (1 if self.c else 0)

    def step(self, stream, ev=None, H=None, ws=None):
        from late_layer_kv_gb300 import ridgefill_fill
        s, d = self.shape, self.d
        if self.c:
            from late_layer_kv_gb300 import RF_RESCALE_VALUES, ridgefill_rescale
            t = self.tail
            if ev is not None:
                ev[-1].record(stream)
            ridgefill_rescale(t["H_tail"], t["X_true"], self.A, d["b"], d["g"], d["Wk"], d["Wv"],
                              self.Kc, self.Vc, which=RF_RESCALE_VALUES, head_dim=s.head_dim,
                              rms_eps=s.rms_eps, rows=0, scale=self.scale,
                              workspace=self.rws, stream=stream, A_scale=self.A_scale)
        ridgefill_fill(self.H_dev if H is None else H, self.A, d["b"], d["g"], d["Wk"], d["Wv"],
                       self.Kc, self.Vc, head_dim=s.head_dim, rope_theta=s.rope_theta,
                       rms_eps=s.rms_eps, rows_per_chunk=self.rpc,
                       workspace=self.ws if ws is None else ws, stream=stream,
                       stage_events=None if ev is None else ev[:3],
                       copy_events=None if (ev is None or not self.host_maps) else
                       ev[3:3 + 2 * s.n_layers], v_scale=self.scale if self.c else None,
                       A_scale=self.A_scale, row_idx=self.row_idx, q8_group_layers=self.q8_group)

    def copy_ms(self, ev):
        """Durations of the first chunk's per-layer map copies (host maps only)."""
        return [ev[3 + 2 * l].elapsed_time(ev[4 + 2 * l]) for l in range(self.shape.n_layers)]

    def stage_ms(self, ev):
        out = {"map_gemm": ev[0].elapsed_time(ev[1]), "kv_gemm": ev[1].elapsed_time(ev[2])}
        if self.c:
            out["value_rescale"] = ev[-1].elapsed_time(ev[0])
        return out

    # end to end: pinned H in, two cache rows per layer out
    def e2e_buffers(self):
        from late_layer_kv_gb300 import ridgefill as rb
        s = self.shape
        self.H_host = self.inp["H"].pin_memory()
        self.out_host = torch.empty((s.n_layers, s.n_kv, 2, s.head_dim),
                                    dtype=torch.bfloat16).pin_memory()
        # the fill reads the pinned split state itself, its copy overlapped with the map GEMM
        # (with a row list the rows are copied first, then gathered)
        self.h_from_host = self.row_idx is None
        if self.h_from_host:
            a = rb.fill_args(self.H_host, self.A, self.d["b"], self.d["g"], self.d["Wk"],
                             self.d["Wv"], self.Kc, self.Vc, head_dim=s.head_dim,
                             rope_theta=s.rope_theta, rms_eps=s.rms_eps, rows_per_chunk=self.rpc,
                             A_scale=self.A_scale)
            self.ws_e2e = torch.empty(rb.fill_workspace_size(a), dtype=torch.uint8,
                                      device=self.Kc.device)
        else:
            self.H_dev = torch.empty_like(self.d["H"])
        bi = self.H_host.numel() * 2
        if self.c:  # the tail rows' split states and true inputs come from the host too
            self.tail_host = {k: v.cpu().pin_memory() for k, v in self.tail.items()}
            bi += sum(v.numel() * 2 for v in self.tail_host.values())
        return bi, self.out_host.numel() * 2

    def e2e_step(self, stream):
        r = self.shape.rows
        if self.c:
            for k, v in self.tail_host.items():
                self.tail[k].copy_(v, non_blocking=True)
        if self.h_from_host:
            self.step(stream, H=self.H_host, ws=self.ws_e2e)
        else:
            self.H_dev.copy_(self.H_host, non_blocking=True)
            self.step(stream)
        self.out_host.copy_(self.Kc[:, :, r - 2:r], non_blocking=True)

    def cpu_rate(self, budget_flop):
        import oracle
        s = self.shape
        per_row = s.n_layers * 2.0 * (s.d * s.d + s.d * 2 * s.kv_width)
        n = int(max(64, min(s.rows, budget_flop / per_row)))
        o = {k: to_f64(v) for k, v in self.inp.items()}
        idx = np.sort(np.random.default_rng(0).choice(s.rows, size=n, replace=False))
        t0 = time.perf_counter()
        oracle.fill_attention(o["H"][idx], idx, o["A"], o["b"], o["g"], o["Wk"], o["Wv"],
                              s.rms_eps, s.rope_theta, s.n_kv, s.head_dim)
        dt = time.perf_counter() - t0
        return (n * s.n_layers / dt, dt,
                f"{n} seeded random prefix rows x all {s.n_layers} late layers")

    def config(self):
        s = self.shape
        return {"workload": s.name, "d": s.d, "late_layers": s.n_layers, "N": s.N, "T": s.T,
                "filled_rows": s.rows, "kv_heads": s.n_kv, "head_dim": s.head_dim,
                "maps": "pinned host, streamed per layer" if self.host_maps else "hbm",
                "map_format": "int8, one bf16 scale per 128 weights" if self.q8 else "bf16",
                "int8_path": (None if not self.q8 else
                              "converted inside the GEMM" if (self.q8_group < 0 or self.host_maps)
                              else f"dequantised {self.q8_group or 4} layers at a time"),
                "rows_per_chunk": self.rpc or s.rows,
                "value_rescale_tail_rows": self.c,
                "exact_prefix_rows": s.rows - self.n_fill,
                "l2": "inputs larger than L2 (maps %d MiB, split state %d MiB)" % (
                    s.n_layers * s.d * s.d * 2 >> 20, s.rows * s.d * 2 >> 20)}


def gdn_state_tensor_flop(rows: int, layers: int, heads: int, chunk: int = 64,
                          d: int = 128) -> float:
    """FLOPs the chunked gated-delta-rule state kernel issues on the tensor cores (one
    (layer, head) state of d x d per CTA, chunks of 64 rows; every product on bf16 high
    and low parts).  Per chunk, in M x N x K shapes of 2 M N K FLOP each:
    P = K K^T: 16 of 128 x 64 x 16 (the stacked [K_hi; K_lo] against K_hi, K_lo);
    U^T: 4 of 128 x 128 x 16 and 4 of 128 x 64 x 16;  W^T: 12 of 128 x 64 x 16;
    NEW^T = U^T - S W^T: 8 of 128 x 128 x 16 and 8 of 128 x 64 x 16;
    S += NEW'^T K: 12 of 128 x 128 x 16."""
    n128 = 4 + 8 + 12          # 128 x 128 x 16 products
    n64 = 16 + 4 + 12 + 8      # 128 x 64 x 16 products
    per_chunk = 2.0 * 16 * d * (n128 * d + n64 * chunk)
    chunks = -(-rows // chunk)
    return per_chunk * chunks * layers * heads


class HybridWorkload:
    """Gated DeltaNet late layers (ridgefill_fill_gdn) plus attention late layers."""

    def __init__(self, shape: GdnShape, exact_frac=0.0):
        self.shape = s = shape
        La, Lg, H = s.n_attn, s.n_gdn, s.n_heads
        kvw = s.n_kv * s.head_dim
        self.exact_frac = exact_frac
        self.n_exact = int(round(exact_frac * s.rows))
        # filled token-layers: exact rows still enter the GDN state but are not filled
        self.token_layers = (s.rows - self.n_exact) * (La + Lg)
        self.stage_names = ["attn_map_gemm", "attn_kv_gemm", "gdn_map_gemm", "gdn_proj_gemm",
                            "gdn_state"]
        proj = H * s.d_k + H * s.d_v + 2 * H
        self.stage_work = {
            "attn_map_gemm": 2.0 * (s.rows - self.n_exact) * La * s.d * s.d,
            "attn_kv_gemm": 2.0 * (s.rows - self.n_exact) * La * s.d * 2 * kvw,
            # with exact rows the GDN map GEMM runs on the filled rows only
            "gdn_map_gemm": 2.0 * (s.rows - self.n_exact) * Lg * s.d * s.d,
            "gdn_proj_gemm": 2.0 * s.rows * Lg * s.d * proj,
            "gdn_state": gdn_state_tensor_flop(s.rows, Lg, H),
        }
        self.stage_bound = {k: "tensor" for k in self.stage_names}
        # the layer's own work counted once: the state as the recurrence's 4 d_v d_k per row
        # and head (the chunked form issues more on the tensor cores, its split products)
        self.total_flops = sum(v for k, v in self.stage_work.items() if k != "gdn_state") + \
            4.0 * s.rows * Lg * H * s.d_v * s.d_k

    def launches_per_step(self):
        # attention map + K/V + RoPE table (+ gather), GDN map, projection, state (+ filled-row
        # list, gather, exact input, rho, finish)
        return 6 + (6 if self.exact_frac else 0)

    def setup(self, dev, seed):
        from late_layer_kv_gb300 import ridgefill as rb
        s = self.shape
        # the library runs the states of the first layers beside the projection GEMM of the
        # rest when all rows fit one chunk and the states outnumber the SMs (one per SM): the
        # "gdn_proj_gemm" stage then holds those states too, and "gdn_state" the last layers'
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        per_wave = sms // s.n_heads
        la = s.n_gdn - per_wave if 0 < per_wave < s.n_gdn else 0
        self.overlap_layers = la
        self.stage_work["gdn_state"] = gdn_state_tensor_flop(s.rows, s.n_gdn - la, s.n_heads)
        self.inp = gdn_inputs(s, seed=seed)
        self.d = {k: v.to(dev) for k, v in self.inp.items()}
        self.Kc = torch.zeros((s.n_attn, s.n_kv, s.N, s.head_dim), dtype=torch.bfloat16,
                              device=dev)
        self.Vc = torch.zeros_like(self.Kc)
        self.S = torch.zeros((s.n_gdn, s.n_heads, s.d_v, s.d_k), dtype=torch.float32, device=dev)
        d = self.d
        a = rb.fill_args(d["H"], d["attn_A"], d["attn_b"], d["attn_g"], d["attn_Wk"],
                         d["attn_Wv"], self.Kc, self.Vc, head_dim=s.head_dim,
                         rope_theta=s.rope_theta, rms_eps=s.rms_eps)
        g = rb.gdn_args(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], d["Wa"], d["Wb"],
                        self.S, n_heads=s.n_heads, rms_eps=s.rms_eps)
        self.row_idx = self.exact_idx = self.X_exact = self.rho = self.dM = None
        if self.exact_frac:
            ex = exact_rows(s.rows, self.exact_frac, seed=seed)
            keep = np.ones(s.rows, bool)
            keep[ex.numpy()] = False
            self.row_idx = torch.from_numpy(np.nonzero(keep)[0].astype(np.int32)).to(dev)
            self.exact_idx = ex.to(dev)
            self.X_exact = true_inputs(s.n_gdn, self.n_exact, s.d, seed=seed).to(dev)
            self.rho = torch.empty((s.n_gdn, s.n_heads), dtype=torch.float32, device=dev)
            gen = torch.Generator(device=dev).manual_seed(seed)
            self.dM = 1e-3 * torch.randn((s.n_gdn, s.n_heads, s.d_v, s.d_k), generator=gen,
                                         device=dev)
            a = rb.fill_args(d["H"], d["attn_A"], d["attn_b"], d["attn_g"], d["attn_Wk"],
                             d["attn_Wv"], self.Kc, self.Vc, head_dim=s.head_dim,
                             rope_theta=s.rope_theta, rms_eps=s.rms_eps, row_idx=self.row_idx)
            g = rb.gdn_args(d["H"], d["A"], d["b"], d["g"], d["Wk"], d["Wv"], d["Wa"], d["Wb"],
                            self.S, n_heads=s.n_heads, rms_eps=s.rms_eps, exact_idx=self.exact_idx,
                            X_exact=self.X_exact, rho=self.rho, delta_M=self.dM)
        self.ws = torch.empty(max(rb.fill_workspace_size(a), rb.gdn_workspace_size(g)),
                              dtype=torch.uint8, device=dev)
        self.H_dev = d["H"]

    def n_events(self):
        return 7

    def step(self, stream, ev=None, H=None, ws=None):
        from late_layer_kv_gb300 import ridgefill_fill, ridgefill_fill_gdn
        s, d = self.shape, self.d
        Hx = self.H_dev if H is None else H
        wsx = self.ws if ws is None else ws
        ridgefill_fill(Hx, d["attn_A"], d["attn_b"], d["attn_g"], d["attn_Wk"],
                       d["attn_Wv"], self.Kc, self.Vc, head_dim=s.head_dim,
                       rope_theta=s.rope_theta, rms_eps=s.rms_eps, workspace=wsx,
                       stream=stream, stage_events=None if ev is None else ev[0:3],
                       row_idx=self.row_idx)
        ridgefill_fill_gdn(Hx, d["A"], d["b"], d["g"], d["Wk"], d["Wv"], d["Wa"],
                           d["Wb"], self.S, n_heads=s.n_heads, rms_eps=s.rms_eps,
                           workspace=wsx, stream=stream,
                           stage_events=None if ev is None else ev[3:7],
                           exact_idx=self.exact_idx, X_exact=self.X_exact, rho=self.rho,
                           delta_M=self.dM)

    def stage_ms(self, ev):
        pairs = [(0, 1), (1, 2), (3, 4), (4, 5), (5, 6)]
        return {n: ev[a].elapsed_time(ev[b]) for n, (a, b) in zip(self.stage_names, pairs)}

    def e2e_buffers(self):
        from late_layer_kv_gb300 import ridgefill as rb
        s, d = self.shape, self.d
        self.H_host = self.inp["H"].pin_memory()
        self.out_host = torch.empty(self.S.shape, dtype=torch.float32).pin_memory()
        # each call reads the pinned split state itself, its copy overlapped with its map
        # GEMM (two copies of H per step); with a row list H is copied once, first
        self.h_from_host = self.row_idx is None
        if self.h_from_host:
            a = rb.fill_args(self.H_host, d["attn_A"], d["attn_b"], d["attn_g"], d["attn_Wk"],
                             d["attn_Wv"], self.Kc, self.Vc, head_dim=s.head_dim,
                             rope_theta=s.rope_theta, rms_eps=s.rms_eps)
            g = rb.gdn_args(self.H_host, d["A"], d["b"], d["g"], d["Wk"], d["Wv"], d["Wa"],
                            d["Wb"], self.S, n_heads=s.n_heads, rms_eps=s.rms_eps,
                            exact_idx=self.exact_idx, X_exact=self.X_exact, rho=self.rho,
                            delta_M=self.dM)
            self.ws_e2e = torch.empty(max(rb.fill_workspace_size(a), rb.gdn_workspace_size(g)),
                                      dtype=torch.uint8, device=self.S.device)
            return 2 * self.H_host.numel() * 2, self.out_host.numel() * 4
        self.H_dev = torch.empty_like(self.d["H"])
        return self.H_host.numel() * 2, self.out_host.numel() * 4

    def e2e_step(self, stream):
        if self.h_from_host:
            self.step(stream, H=self.H_host, ws=self.ws_e2e)
        else:
            self.H_dev.copy_(self.H_host, non_blocking=True)
            self.step(stream)
        self.out_host.copy_(self.S, non_blocking=True)

    def cpu_rate(self, budget_flop):
        """Attention layers on sampled rows, GDN layers on the first rows of one layer
        (its state needs every earlier row); combined per token-layer in the layer mix."""
        import oracle
        s = self.shape
        o = {k: to_f64(v) for k, v in self.inp.items()}
        kvw = s.n_kv * s.head_dim
        per_row = s.n_attn * 2.0 * (s.d * s.d + s.d * 2 * kvw)
        na = int(max(64, min(s.rows, budget_flop / 2 / per_row)))
        idx = np.sort(np.random.default_rng(0).choice(s.rows, size=na, replace=False))
        t0 = time.perf_counter()
        oracle.fill_attention(o["H"][idx], idx, o["attn_A"], o["attn_b"], o["attn_g"],
                              o["attn_Wk"], o["attn_Wv"], s.rms_eps, s.rope_theta, s.n_kv,
                              s.head_dim)
        ta = (time.perf_counter() - t0) / (na * s.n_attn)
        ng = 256
        t0 = time.perf_counter()
        oracle.gdn_state(o["H"][:ng], o["A"], o["b"], o["g"], o["Wk"], o["Wv"], o["Wa"], o["Wb"],
                         s.rms_eps, s.n_heads, s.d_k, s.d_v, layers=[0])
        tg = (time.perf_counter() - t0) / ng
        per = (s.n_attn * ta + s.n_gdn * tg) / (s.n_attn + s.n_gdn)
        return 1.0 / per, na * s.n_attn * ta + ng * tg, (
            f"attention: {na} random prefix rows x {s.n_attn} layers; GDN: first {ng} rows x 1 "
            f"layer x {s.n_heads} heads; combined per token-layer in the "
            f"{s.n_attn}:{s.n_gdn} mix")

    def config(self):
        s = self.shape
        return {"workload": s.name, "d": s.d, "late_layers": s.n_attn + s.n_gdn,
                "gdn_layers": s.n_gdn, "attn_layers": s.n_attn, "gdn_heads": s.n_heads,
                "d_k": s.d_k, "d_v": s.d_v, "N": s.N, "T": s.T, "filled_rows": s.rows - self.n_exact,
                "exact_prefix_rows": self.n_exact,
                "terminal_correction": bool(self.exact_frac),
                "kv_heads": s.n_kv, "head_dim": s.head_dim, "maps": "hbm",
                "gdn_states_beside_projection": getattr(self, "overlap_layers", 0),
                "l2": "inputs larger than L2 (maps %d MiB)" % (
                    (s.n_attn + s.n_gdn) * s.d * s.d * 2 >> 20)}


class FitWorkload:
    """The ridge fit of every late layer's map from calibration pairs (ridgefill_fit):
    one accumulate call over all calibration rows, then the solve."""

    metric = "ridge fit: calibration row-layers/s (accumulate + solve of every late map)"
    unit = "row-layers/s"

    def __init__(self, shape: FillShape, rows: int):
        self.shape, self.n = shape, rows
        s = shape
        L, d = s.n_layers, s.d
        self.token_layers = rows * L  # calibration row-layers per fit
        self.stage_names = ["accumulate", "solve"]
        self.stage_work = {"accumulate": 2.0 * rows * d * (d + L * d),
                           "solve": 2.0 * L * d * 3 * d * d}
        self.stage_bound = {"accumulate": "tensor", "solve": "tensor"}
        self.total_flops = sum(self.stage_work.values())

    def launches_per_step(self):
        d = self.shape.d
        nb = d // 64
        # triangular inverse by recursive doubling: per part of a level four operand splits
        # and two batched products
        inv, sz = 0, 64
        while sz < d:
            full = d // (2 * sz)
            rest = d - full * 2 * sz
            inv += 6 * ((1 if full > 0 else 0) + (1 if rest > sz else 0))
            sz *= 2
        # accumulate: two column-sum passes, their reduction, the count, the Gram products;
        # solve: preparation, equilibration, Cholesky (the first diagonal block, then per
        # step a panel launch that also factors the next diagonal block and, while columns
        # from four blocks on remain, the trailing update; the last held-back block's copy),
        # zero fill, the doubling products, the bf16 split, the G^-1 product, two operand
        # splits, the solve GEMM, the offsets
        chol = 1 + (nb - 1) + max(0, nb - 4) + (1 if nb > 1 else 0)
        return 5 + 2 + chol + 1 + inv + 1 + 1 + 2 + 1 + 1

    def setup(self, dev, seed):
        """Calibration pairs drawn on the device (synthetic.calibration_device)."""
        from late_layer_kv_gb300 import FitSums
        from late_layer_kv_gb300 import ridgefill as rb
        s, n = self.shape, self.n
        L, d = s.n_layers, s.d
        cal = calibration_device(d, L, n, seed, dev)
        self.X, self.Y = cal["X"], cal["Y"]
        self.sums = FitSums(L, d, d, device=dev)
        self.A = torch.empty((L, d, d), dtype=torch.bfloat16, device=dev)
        self.b = torch.empty((L, d), dtype=torch.float32, device=dev)
        a = rb.FitArgs(L, d, d, rb.RF_FIT_SOLVE, 0, s.lam)
        self.ws = torch.empty(int(rb.load().ridgefill_fit_workspace_size(ctypes_byref(a))),
                              dtype=torch.uint8, device=dev)

    def n_events(self):
        return 3

    def step(self, stream, ev=None):
        from late_layer_kv_gb300 import ridgefill_fit_accumulate, ridgefill_fit_solve
        for t in (self.sums.G, self.sums.C, self.sums.sx, self.sums.sy, self.sums.count):
            t.zero_()
        if ev is not None:
            ev[0].record(stream)
        ridgefill_fit_accumulate(self.sums, self.X, self.Y, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        ridgefill_fit_solve(self.sums, self.shape.lam, A_out=self.A, b_out=self.b,
                            workspace=self.ws, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    def stage_ms(self, ev):
        return {"accumulate": ev[0].elapsed_time(ev[1]), "solve": ev[1].elapsed_time(ev[2])}

    # e2e: the calibration pairs come from pinned host memory in row batches, each copied
    # on a side stream into one of two device buffers while the previous batch is added to
    # the sums (the running sums are additive over batches); then the solve, and the maps
    # are read back.
    E2E_BATCHES = 8

    def e2e_buffers(self):
        s, n = self.shape, self.n
        self.X_host = self.X.cpu().pin_memory()
        self.Y_host = self.Y.cpu().pin_memory()
        self.A_host = torch.empty(self.A.shape, dtype=torch.bfloat16).pin_memory()
        nbat = self.E2E_BATCHES if n % self.E2E_BATCHES == 0 else 1
        self.rb = n // nbat
        dev = self.X.device
        self.Xb = [torch.empty((self.rb, s.d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.Yb = [torch.empty((s.n_layers, self.rb, s.d), dtype=torch.bfloat16, device=dev)
                   for _ in range(2)]
        self.cstream = torch.cuda.Stream(dev)
        self.copied = [torch.cuda.Event() for _ in range(2)]
        self.used = [torch.cuda.Event() for _ in range(2)]
        return (self.X_host.numel() + self.Y_host.numel()) * 2, self.A_host.numel() * 2

    def e2e_step(self, stream):
        from late_layer_kv_gb300 import ridgefill_fit_accumulate, ridgefill_fit_solve
        for t in (self.sums.G, self.sums.C, self.sums.sx, self.sums.sy, self.sums.count):
            t.zero_()
        rb = self.rb
        for i, r0 in enumerate(range(0, self.n, rb)):
            k = i % 2
            self.cstream.wait_event(self.used[k])  # buffer k's previous batch was added
            with torch.cuda.stream(self.cstream):
                self.Xb[k].copy_(self.X_host[r0:r0 + rb], non_blocking=True)
                for l in range(self.shape.n_layers):
                    self.Yb[k][l].copy_(self.Y_host[l, r0:r0 + rb], non_blocking=True)
                self.copied[k].record(self.cstream)
            stream.wait_event(self.copied[k])
            ridgefill_fit_accumulate(self.sums, self.Xb[k], self.Yb[k], stream=stream)
            self.used[k].record(stream)
        ridgefill_fit_solve(self.sums, self.shape.lam, A_out=self.A, b_out=self.b,
                            workspace=self.ws, stream=stream)
        self.A_host.copy_(self.A, non_blocking=True)

    def cpu_rate(self, budget_flop):
        """The f64 oracle fit of one layer on a row sample of the calibration pairs."""
        import oracle
        d = self.shape.d
        n = int(max(256, min(self.n, budget_flop / (4.0 * d * d))))
        X = to_f64(self.X[:n].cpu())
        Y = to_f64(self.Y[:1, :n].cpu())
        t0 = time.perf_counter()
        oracle.ridge_fit(X, Y, self.shape.lam)
        dt = time.perf_counter() - t0
        return n / dt, dt, f"one layer's fit from the first {n} calibration rows (row-layers/s)"

    def config(self):
        s = self.shape
        return {"workload": s.name + "_fit", "d": s.d, "late_layers": s.n_layers,
                "calibration_rows": self.n, "lambda": s.lam,
                "l2": "inputs larger than L2 (calibration pairs %d MiB)" % (
                    self.n * s.d * (s.n_layers + 1) * 2 >> 20)}


def ctypes_byref(x):
    import ctypes
    return ctypes.byref(x)


def make_workload(name, args):
    if args.fit:
        shape = WORKLOADS[name]
        return FitWorkload(shape, args.fit_rows or shape.calib_rows)
    shape = WORKLOADS[name]
    if isinstance(shape, GdnShape):
        if args.rows:
            shape = replace(shape, name=f"{shape.name}_rows{args.rows}", N=args.rows + shape.T)
        return HybridWorkload(shape, exact_frac=args.exact_frac)
    if args.rows or args.layers:
        rows = args.rows or shape.rows
        L = args.layers or shape.n_layers
        shape = replace(shape, name=f"{shape.name}_rows{rows}_L{L}", N=rows + shape.T, n_layers=L)
    rpc = args.rows_per_chunk
    if name.startswith("dense27b") and not rpc:
        rpc = 16384  # late-layer X_hat processed in row chunks
    return AttnWorkload(shape, host_maps=name.startswith("hostmaps"), rows_per_chunk=rpc,
                        rescale_rows=args.rescale, int8_maps=args.int8_maps,
                        q8_group=args.q8_group,
                        exact_frac=args.exact_frac)


# ----------------------------------------------------------------------------- arms

def _copy_ms(dst, src):
    e0, e1 = _events(2)
    e0.record()
    dst.copy_(src, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def h2d_rate_gbs(dev, nbytes=32 << 20, reps=20):
    """Best-of pinned host -> device copy rate (GB/s)."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(reps + 3):
        e0, e1 = _events(2)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1000.0) / 1e9)
    return best


def _measure(wl, stream, steps, warmup, world, dev, local):
    """Warm-up, then `steps` timed steps bracketed by a barrier and a device sync, with
    the library's stage events per step and nvidia-smi clocks sampled meanwhile.
    Returns (timed-region ms, the max over ranks; per-step events; clocks)."""
    from late_layer_kv_gb300 import device_error
    ev = [_events(wl.n_events()) for _ in range(steps)]
    for e in sum(ev, []):
        e.record(stream)  # torch creates the CUDA event on first record
    for _ in range(warmup):
        wl.step(stream)
    torch.cuda.synchronize()
    assert device_error(stream) == 0, "device wait ran out during warm-up"
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0, t1 = _events(2)
    t0.record(stream)
    for i in range(steps):
        wl.step(stream, ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    assert device_error(stream) == 0, "device wait ran out during the timed region"
    return max_over_ranks(t0.elapsed_time(t1), world, dev), ev, clk


def _stages(wl, ev, ms):
    """Per-stage mean ms, achieved TFLOP/s and fraction of the bf16 peak (burst for timed
    regions under 2 s, sustained otherwise), and the dominant stage's roofline."""
    peaks, src = _peaks()
    pkey = "bf16_tflops_sustained" if ms >= 2000.0 else "bf16_tflops"
    tpeak = float(peaks[pkey])
    stages = {}
    for name in wl.stage_names:
        sm = float(np.mean([wl.stage_ms(e)[name] for e in ev]))
        ach = wl.stage_work[name] / (sm / 1000.0) / 1e12
        stages[name] = {"ms": sm, "achieved_tflops": ach, "bound": wl.stage_bound[name],
                        "frac": ach / tpeak}
    dom = max(stages, key=lambda k: stages[k]["ms"])
    traffic = None
    pt = PROFILED_TRAFFIC.get(wl.config()["workload"])
    if pt and pt["kernel_sha256"] == _kernel_digest(pt["sources"]):
        traffic = pt["bytes_per_launch"]
    roofline = {"bound": stages[dom]["bound"], "kernel": dom,
                "achieved": stages[dom]["achieved_tflops"], "peak": tpeak, "unit": "TFLOP/s",
                "frac": stages[dom]["achieved_tflops"] / tpeak, "traffic": traffic,
                "peak_source": f"{src} {pkey}", "timed_region_ms": ms}
    return stages, roofline, tpeak


def _host_link(wl, ev, stages, dev):
    """Map-copy rates of a host-map fill against the measured pinned host-to-device link."""
    s = wl.shape
    link = h2d_rate_gbs(dev)
    # bytes per layer on the link: bf16 maps, or int8 codes plus bf16 scales
    layer_bytes = s.d * s.d * 2 if not wl.q8 else s.d * s.d + s.d * (s.d // 128) * 2
    map_bytes = s.n_layers * layer_bytes
    mstage = stages["map_gemm"]["ms"]
    cms = [t for e in ev for t in wl.copy_ms(e)]
    # median per copy: the pool's host link shows stalls of tens of ms from other tenants,
    # which the mean (also reported) takes in
    copy_gbs = layer_bytes / (float(np.median(cms)) / 1000.0) / 1e9
    copy_gbs_mean = layer_bytes / (float(np.mean(cms)) / 1000.0) / 1e9
    one = wl.A[0].view(-1)  # the maps' own pinned buffer, alone on the link
    tmp = torch.empty_like(one, device=dev)
    maps_buf = max(one.numel() * one.element_size() / (t / 1000.0) / 1e9 for t in
                   [_copy_ms(tmp, one) for _ in range(10)])
    return {"h2d_gbs_measured": link, "maps_buffer_h2d_gbs": maps_buf,
            "map_bytes_per_step": map_bytes,
            "copy_gbs": copy_gbs, "copy_gbs_mean": copy_gbs_mean,
            "copy_frac_of_link": copy_gbs / link,
            "map_stage_gbs": map_bytes / (mstage / 1000.0) / 1e9,
            "note": "maps copied per layer on a side stream while the previous layer "
                    "computes; copy_gbs is the median rate of those copies (events on "
                    "the copy stream), copy_gbs_mean their mean, map_stage_gbs the rate "
                    "the maps flowed through the map stage"}


def _secondary(args, head, dev, stream, local):
    """The other workloads, each timed on its own (CUDA events on the launching stream,
    its own warm-up and clocks): maps streamed from host memory at both prompt lengths, the
    hybrid Gated DeltaNet fill, the 27B-class fill at all four prompt lengths, and the fit."""
    out = {}

    def run(name, wl, steps, setup):
        t = time.perf_counter()
        setup(wl)
        ms, ev, clk = _measure(wl, stream, steps, max(3, min(args.warmup, 5)), 1, dev, local)
        stages, roof, _ = _stages(wl, ev, ms)
        ms_step = ms / steps
        e = {"config": wl.config(), "steps": steps, "ms_per_step": ms_step,
             "value": wl.token_layers / (ms_step / 1000.0),
             "unit": getattr(wl, "unit", "token-layers/s"),
             "pct_bf16_peak": 100.0 * wl.total_flops / (ms_step / 1000.0) / 1e12 / roof["peak"],
             "stages": stages, "roofline": roof, "clocks": clk,
             "gpu_launches": wl.launches_per_step() * steps}
        if getattr(wl, "host_maps", False):
            e["host_link"] = _host_link(wl, ev, stages, dev)
        e["wall_s"] = time.perf_counter() - t
        out[name] = e
        return wl

    seed = 1001
    # maps streamed from pinned host memory: the headline's inputs at 16K, then the 64K prompt
    for name, steps, inp in (("hostmaps_16k", 20, head.inp), ("hostmaps_64k", 10, None)):
        wl = run(name, AttnWorkload(WORKLOADS[name], host_maps=True), min(args.steps, steps),
                 lambda w, inp=inp: w.setup(dev, seed, inp=inp))
        del wl
        torch.cuda.empty_cache()
    wl = run("hybrid_gdn_32k", HybridWorkload(WORKLOADS["hybrid_gdn_32k"]),
             min(args.steps, 20), lambda w: w.setup(dev, seed))
    del wl
    torch.cuda.empty_cache()
    # the 27B-class sweep: one draw at the longest prompt, whose first rows serve the shorter
    big = fill_inputs(WORKLOADS["dense27b_120k"], seed=seed)
    for name, steps in (("dense27b_120k", 5), ("dense27b_64k", 8), ("dense27b_32k", 10),
                        ("dense27b_16k", 20)):
        inp = dict(big)
        inp["H"] = big["H"][:WORKLOADS[name].rows]
        wl = run(name, AttnWorkload(WORKLOADS[name], rows_per_chunk=16384), min(args.steps, steps),
                 lambda w, inp=inp: w.setup(dev, seed, inp=inp))
        del wl, inp
        torch.cuda.empty_cache()
    del big
    shape = WORKLOADS["hostmaps_16k"]
    wl = run("fit", FitWorkload(shape, shape.calib_rows), min(args.steps, 10),
             lambda w: w.setup(dev, seed))
    del wl
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = make_workload(args.workload, args)
    wl.setup(dev, seed=1001 + rank)
    stream = torch.cuda.current_stream(dev)
    steps = args.steps
    ms, ev, clk = _measure(wl, stream, steps, args.warmup, world, dev, local)
    ms_step = ms / steps
    value = whole_job_rate(wl.token_layers, world, ms_step)
    stages, roofline, tpeak = _stages(wl, ev, ms)
    pct = 100.0 * wl.total_flops / (ms_step / 1000.0) / 1e12 / tpeak

    e2e = None
    if not args.no_e2e:
        bi, bo = wl.e2e_buffers()
        for _ in range(3):
            wl.e2e_step(stream)
        torch.cuda.synchronize()
        e0, e1 = _events(2)
        e0.record(stream)
        for _ in range(steps):
            wl.e2e_step(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1) / steps, world, dev)
        e2e = {"value": whole_job_rate(wl.token_layers, world, ems), "unit": getattr(wl, "unit", "token-layers/s"),
               "ms_per_step": ems, "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
               "note": "H copied from pinned host memory inside the timed region; the caches "
                       "stay on the device (their consumer is the exact tail's attention), "
                       "two cache rows per layer are read back" if isinstance(wl, AttnWorkload)
                       else None}

    host_link = None
    if getattr(wl, "host_maps", False):
        host_link = _host_link(wl, ev, stages, dev)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        r, dt, what = wl.cpu_rate(args.cpu_flop)
        cpu = {"value": r, "unit": getattr(wl, "unit", "token-layers/s"), "cores": _cores(), "kind": "oracle",
               "sample": f"{what} ({dt:.1f} s of f64 numpy work)"}

    secondary = None
    plain = (args.workload == "llama8b_16k" and not (args.fit or args.rows or args.layers or
             args.rows_per_chunk or args.exact_frac or args.int8_maps or args.rescale))
    if world == 1 and plain and not args.no_secondary:
        secondary = _secondary(args, wl, dev, stream, local)

    if rank == 0:
        line = {
            "metric": getattr(wl, "metric", METRIC), "value": value, "unit": getattr(wl, "unit", "token-layers/s"), "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": wl.config(),
            "fill_stage_ms": ms_step, "pct_bf16_peak": pct, "stages": stages,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": wl.launches_per_step() * steps, "clocks": clk,
        }
        if host_link:
            line["host_link"] = host_link
        if secondary:
            line["secondary"] = secondary
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The oracle as it stands, on the host cores, for the same metric and workload."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    if args.fit:
        print(json.dumps({"impl": "reference", "unavailable": "the fit line has no reference arm"}))
        return
    wl = make_workload(args.workload, args)
    wl.inp = (gdn_inputs(wl.shape, seed=1001) if isinstance(wl, HybridWorkload)
              else fill_inputs(wl.shape, seed=1001))
    rates, times, what = [], [], ""
    for i in range(args.warmup + args.steps):
        r, dt, what = wl.cpu_rate(args.ref_flop)
        if i >= args.warmup:
            rates.append(r)
            times.append(dt)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "token-layers/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * float(np.mean(times)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": wl.config(),
        "cpu_baseline": {"value": value, "unit": "token-layers/s", "cores": _cores(),
                         "kind": "oracle", "sample": what + " per step"},
        "e2e": {"value": value, "unit": "token-layers/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="llama8b_16k", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-flop", type=float, default=6e12,
                    help="f64 work of the CPU-baseline sample (about 10-30 s on the host)")
    ap.add_argument("--ref-flop", type=float, default=2e11,
                    help="f64 work per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="default workload: skip the other workloads timed after the headline")
    ap.add_argument("--rows", type=int, default=0, help="override the filled rows (profiling)")
    ap.add_argument("--layers", type=int, default=0, help="override the late layers (profiling)")
    ap.add_argument("--rows-per-chunk", type=int, default=0)
    ap.add_argument("--fit", action="store_true",
                    help="benchmark the ridge fit of the workload's maps instead of the fill")
    ap.add_argument("--fit-rows", type=int, default=0)
    ap.add_argument("--exact-frac", type=float, default=0.0,
                    help="share of prefix rows run exactly (skipped by the fill; GDN layers take "
                         "their true inputs and apply the terminal-state correction)")
    ap.add_argument("--int8-maps", action="store_true",
                    help="maps as int8 codes with one bf16 scale per 128 weights")
    ap.add_argument("--q8-group", type=int, default=0, metavar="K",
                    help="resident int8 maps: layers dequantised at a time ahead of the bf16 "
                         "GEMM (0: the library's 4; -1: converted inside the GEMM)")
    ap.add_argument("--rescale", type=int, default=0, metavar="C",
                    help="also apply the value rescale from C exact tail rows each step")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
