#!/usr/bin/env python
"""Benchmark of the GGML dequant-GEMV hot path on one GB300 (one JSON line on stdout).

Workload of the headline line ("q8_0_decode_3072x8192_28L"): 28 layers of
batch-1 Q8_0 GEMVs, each layer an up projection 3072 -> 8192 and a down
projection 8192 -> 3072 (distinct random matrices, 1.50 GB in total, cycled
so no weight is L2-resident).  One step = one pass over the 28 layers (56
GEMVs, the up output feeding the down input), captured once in a CUDA graph
and replayed.  value = algorithmic bytes (GGML weight bytes + x + y) per
second over all ranks.

Also measured in the same run (the "rows" object): Q4_K GEMV 3072 -> 8192
(28 copies), the fused Q4_K FFN block with residual (28 layers), the
tensor-core batch GEMM at M = 16 / 64 / 512 for both shapes, and the 256 x 512
Q8_0 GEMV (L2-resident, microseconds only).

--impl reference times the CPU oracle on a bounded sample of the same
workload (rows of the same matrices), on this machine's host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "batch-1 dequant-GEMV weight GB/s & µs/matrix (% of GB300 HBM peak)"
N_EMBD, N_FF, N_LAYERS = 3072, 8192, 28
Q8_W_BYTES = N_FF * N_EMBD // 32 * 34            # 26,738,688
Q4_W_BYTES = N_FF * N_EMBD // 256 * 144          # 14,155,776
GEMV_IO_BYTES = (N_EMBD + N_FF) * 4              # x read + y written
WORKLOAD = "q8_0_decode_3072x8192_28L"


# ---------------------------------------------------------------- host utilities

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# CUDA sources that define each profiled kernel (a recorded counter is stale once any of them changes)
KERNEL_SOURCES = {
    "q8_0_gemv": ["qdq_gemv_xs.cu", "qdq_internal.cuh"],
    "q4k_ffn": ["qdq_gemv_xs.cu", "qdq_internal.cuh"],
}


def kernel_sources_digest(case: str) -> str:
    """sha256 over the CUDA sources of one profiled kernel, in the listed order."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ggml_quantized_dequant_gb300", "csrc")
    for name in KERNEL_SOURCES[case]:
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(case: str):
    """DRAM bytes per launch that ncu measured for `case`, or None if not captured for these sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(case)
    if not d or d.get("sources_sha256") != kernel_sources_digest(case):
        return None
    return float(d["dram_bytes_per_launch"])


def job_value(units_per_rank: float, world: int, t_max_s: float) -> float:
    """Whole-job throughput: every rank processed `units_per_rank`; the job took the slowest rank's time."""
    return units_per_rank * world / t_max_s


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None

    @staticmethod
    def gpu_id(torch, local_rank: int) -> str:
        """nvidia-smi's id for the CUDA device in use (its UUID when torch exposes one)."""
        try:
            u = str(torch.cuda.get_device_properties(local_rank).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            return vis.split(",")[local_rank] if vis else str(local_rank)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            p = [s.strip() for s in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
                power.append(float(p[3]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": float(max(power))}


# ---------------------------------------------------------------- CPU oracle legs

def oracle_rate(n_rows: int, seconds_budget: float):
    """Time the CPU oracle (dequant + float64 GEMV) on row samples of config-1 matrices.

    Returns (bytes_per_s, rows_done, seconds, matrices_rows).  The sample is the
    first `n_rows` rows of layer 0's up and down matrices, repeated until the
    budget is spent; bytes are the sampled rows' GGML weight bytes plus x and y.
    """
    import oracle
    import synth
    up, down = synth.config1_up(0), synth.config1_down(0)
    x_up = synth.config1_x()
    x_dn = synth.activations(synth.rng_for(1, 3), 1, N_FF)
    done_bytes, done_rows, t_used = 0, 0, 0.0
    while t_used < seconds_budget:
        for w, n_in, x in ((up, N_EMBD, x_up), (down, N_FF, x_dn)):
            t0 = time.perf_counter()
            wd = oracle.q8_0_dequant(w[:n_rows], n_rows, n_in)
            oracle.gemv(wd, x)
            t_used += time.perf_counter() - t0
            done_bytes += n_rows * (n_in // 32 * 34) + n_in * 4 + n_rows * 4
            done_rows += n_rows
    return done_bytes / t_used, done_rows, t_used


def cpu_baseline(budget_s: float = 12.0):
    rate, rows, secs = oracle_rate(512, budget_s)
    return {"value": rate / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "CPU oracle (numpy: own fp16 decode, f32 dequant, float64 GEMV, one thread) on the first "
                      "512 rows of config-1 layer-0 up (3072->8192) and down (8192->3072) Q8_0 matrices, "
                      "%d rows in %.1f s" % (rows, secs)}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return 0
    # size each step so the whole --warmup + --steps run takes about a minute
    per_step_s = max(0.01, 60.0 / max(1, args.steps + args.warmup))
    import oracle
    import synth
    up, down = synth.config1_up(0), synth.config1_down(0)
    x_up = synth.config1_x()
    x_dn = synth.activations(synth.rng_for(1, 3), 1, N_FF)
    # calibrate rows per step from a 64-row probe
    t0 = time.perf_counter()
    oracle.gemv(oracle.q8_0_dequant(up[:64], 64, N_EMBD), x_up)
    oracle.gemv(oracle.q8_0_dequant(down[:64], 64, N_FF), x_dn)
    per_row = (time.perf_counter() - t0) / 128
    rows = int(max(2, min(N_EMBD, per_step_s / per_row / 2)))

    def step(i):
        r0 = (i * rows) % (N_EMBD - rows + 1)
        oracle.gemv(oracle.q8_0_dequant(up[r0:r0 + rows], rows, N_EMBD), x_up)
        oracle.gemv(oracle.q8_0_dequant(down[r0:r0 + rows], rows, N_FF), x_dn)
        return rows * (N_EMBD // 32 * 34 + N_FF // 32 * 34) + (N_EMBD + N_FF) * 4 + 2 * rows * 4

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    nbytes = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    gbs = nbytes / dt / 1e9
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "sample_rows_per_matrix_per_step": rows, "batch": 1,
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "%d rows of the config-1 up and down matrices per step (CPU oracle, one thread)"
                                   % rows},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU legs

class Timer:
    """CUDA-event timing on the current stream, with device syncs around it."""

    def __init__(self, torch):
        self.torch = torch

    def __call__(self, fn, iters: int) -> float:
        torch = self.torch
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(iters):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / 1e3


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # one eager run on the capture stream (also warms up)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def gen_parallel(fns):
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        return list(ex.map(lambda f: f(), fns))


def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import synth
    import ggml_quantized_dequant_gb300 as qdq
    from ggml_quantized_dequant_gb300 import _build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        _build.build()
    barrier()
    qdq.load()
    peaks = measured_peaks()
    timer = Timer(torch)

    # ---------------- config 1: 28 layers of Q8_0 up/down ----------------
    ups = gen_parallel([lambda t=t: synth.config1_up(t) for t in range(N_LAYERS)])
    W_up = [qdq.upload_q8_0(w, N_FF, N_EMBD, device=dev) for w in ups]
    del ups
    downs = gen_parallel([lambda t=t: synth.config1_down(t) for t in range(N_LAYERS)])
    W_dn = [qdq.upload_q8_0(w, N_EMBD, N_FF, device=dev) for w in downs]
    del downs
    x_host = synth.config1_x()
    x = torch.from_numpy(x_host).to(dev)
    h = torch.empty((1, N_FF), device=dev)
    y = torch.empty((1, N_EMBD), device=dev)

    def step():
        for t in range(N_LAYERS):
            qdq.q8_0_gemv(W_up[t], x, h, N_FF, N_EMBD, 1)
            qdq.q8_0_gemv(W_dn[t], h, y, N_EMBD, N_FF, 1)

    g = capture(torch, step)
    launches_per_step = 2 * N_LAYERS
    bytes_per_launch = Q8_W_BYTES + GEMV_IO_BYTES
    bytes_per_step = launches_per_step * bytes_per_launch

    # warm clocks (>= 200 ms of work), then the untimed warm-up steps
    t_end = time.time() + 0.3
    while time.time() < t_end:
        g.replay()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()

    barrier()
    torch.cuda.synchronize()
    with ClockSampler(ClockSampler.gpu_id(torch, local_rank)) as clk:
        dt = timer(g.replay, args.steps)
    barrier()
    t_max = reduce_max(dt, dev)
    value_gbs = job_value(bytes_per_step * args.steps, world, t_max) / 1e9
    us_per_matrix = t_max / (args.steps * launches_per_step) * 1e6
    launch_s = t_max / (args.steps * launches_per_step)
    achieved = bytes_per_launch / launch_s / 1e9

    # ---------------- e2e: public API calls, pinned host x in, host y out, every step ----------------
    x_pin = torch.from_numpy(x_host).pin_memory()
    y_pin = torch.empty((1, N_EMBD), dtype=torch.float32).pin_memory()
    x_e = torch.empty_like(x)
    e2e_steps = max(20, min(400, args.steps // 10))

    def e2e_step():
        x_e.copy_(x_pin, non_blocking=True)
        for t in range(N_LAYERS):
            qdq.q8_0_gemv(W_up[t], x_e, h, N_FF, N_EMBD, 1)
            qdq.q8_0_gemv(W_dn[t], h, y, N_EMBD, N_FF, 1)
        y_pin.copy_(y, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(5):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_dt = reduce_max(time.perf_counter() - t0, dev)
    e2e_gbs = job_value(bytes_per_step * e2e_steps, world, e2e_dt) / 1e9

    rows = {}
    if not args.no_rows:
        # the same chain on the opt-in block fixed-point arithmetic (QDQ_OPT_XS_FLOAT_X = 0),
        # whose error bound is relative to each block's largest activation: reported
        # beside the headline, never as it
        old = qdq.set_option(qdq.QDQ_OPT_XS_FLOAT_X, 0)
        try:
            gf = capture(torch, step)
            for _ in range(5):
                gf.replay()
            it = max(20, args.row_steps)
            dtf = timer(gf.replay, it)
        finally:
            qdq.set_option(qdq.QDQ_OPT_XS_FLOAT_X, old)
        usf = dtf / (it * launches_per_step) * 1e6
        rows["q8_0_decode_28L_fixed_point_optin"] = {
            "us_per_matrix": usf, "gbs": bytes_per_launch / usf / 1e3,
            "frac_hbm": bytes_per_launch / usf / 1e3 / peaks["hbm_gbs"],
            "arithmetic": "opt-in block fixed point (bound relative to each block's max |x|, not 1e-5 sum|w||x|)"}
        del gf
        rows.update(measure_rows(torch, qdq, synth, dev, timer, peaks, args))
    del W_up, W_dn

    line = {
        "metric": METRIC, "value": value_gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "layers": N_LAYERS, "shapes": "up 3072->8192, down 8192->3072",
                   "format": "GGML Q8_0", "us_per_matrix": us_per_matrix,
                   "frac_of_hbm_peak": value_gbs / world / peaks["hbm_gbs"],
                   "l2": "inputs larger than L2: 56 distinct matrices, 1.50 GB, cycled every step",
                   "timing": "CUDA graph of one step (56 launches, programmatic dependent launch), "
                             "replayed; CUDA events on the replay stream",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "gemv_xs_kernel<0, 0, 1> (Q8_0 batch-1 GEMV, f32 arithmetic)", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": args.traffic if args.traffic is not None else recorded_traffic("q8_0_gemv"),
                     "peak_source": peaks["source"],
                     "bytes_per_launch": bytes_per_launch},
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": N_EMBD * 4, "d2h_bytes_per_step": N_EMBD * 4,
                "steps": e2e_steps, "ms_per_step": e2e_dt / e2e_steps * 1e3,
                "path": "Python binding -> C ABI per GEMV (no graph), pinned H2D of x and D2H of y each step"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "rows": rows,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    return 0


def measure_rows(torch, qdq, synth, dev, timer, peaks, args):
    """Every hot-path row on its own workload; each returns microseconds per call and its roofline fraction."""
    rows = {}
    iters = max(20, args.row_steps)
    hbm = peaks["hbm_gbs"]

    # config 0: 256 x 512 Q8_0 (L2-resident; microseconds only)
    wb, x0 = synth.config0()
    W0 = qdq.upload_q8_0(wb, 256, 512, device=dev)
    x0d = torch.from_numpy(x0).to(dev)
    y0 = torch.empty((1, 256), device=dev)
    g0 = capture(torch, lambda: [qdq.q8_0_gemv(W0, x0d, y0, 256, 512, 1) for _ in range(100)])
    g0.replay()
    dt = timer(g0.replay, iters)
    rows["q8_0_gemv_256x512"] = {"us_per_call": dt / (iters * 100) * 1e6, "roofline": "n/a (L2-resident)"}

    # config 2: Q4_K 3072 -> 8192, 28 copies cycled
    ws = gen_parallel([lambda t=t: synth.config2_w(t) for t in range(N_LAYERS)])
    W2 = [qdq.upload_q4k(w, N_FF, N_EMBD, device=dev) for w in ws]
    del ws
    x2 = torch.from_numpy(synth.config2_x()).to(dev)
    y2 = torch.empty((1, N_FF), device=dev)
    g2 = capture(torch, lambda: [qdq.q4k_gemv(W2[t], x2, y2, N_FF, N_EMBD, 1) for t in range(N_LAYERS)])
    for _ in range(5):
        g2.replay()
    dt = timer(g2.replay, iters)
    us = dt / (iters * N_LAYERS) * 1e6
    b = Q4_W_BYTES + (N_EMBD + N_FF) * 4
    rows["q4k_gemv_3072x8192"] = {"us_per_call": us, "gbs": b / us / 1e3, "frac_hbm": b / us / 1e3 / hbm,
                                  "bytes_per_call": b}
    del W2

    # config 3: fused Q4_K FFN block with residual, 28 layers
    layers = gen_parallel([lambda t=t: synth.config3_layer(t) for t in range(N_LAYERS)])
    L = [(qdq.upload_q4k(g, N_FF, N_EMBD, device=dev), qdq.upload_q4k(u, N_FF, N_EMBD, device=dev),
          qdq.upload_q4k(d, N_EMBD, N_FF, device=dev)) for g, u, d in layers]
    del layers
    xh, rh = synth.config3_x_residual()
    x3, r3 = torch.from_numpy(xh).to(dev), torch.from_numpy(rh).to(dev)
    mid = torch.empty((1, N_FF), device=dev)

    def ffn_step():
        for Wg, Wu, Wd in L:
            qdq.q4k_ffn_residual(Wg, Wu, Wd, x3, r3, r3, mid, N_EMBD, N_FF, 1)

    g3 = capture(torch, ffn_step)
    for _ in range(5):
        g3.replay()
    dt = timer(g3.replay, iters)
    us = dt / (iters * N_LAYERS) * 1e6
    b = 3 * Q4_W_BYTES + N_EMBD * 4 + N_FF * 4 * 2 + N_EMBD * 4 * 2
    rows["q4k_ffn_residual_3072x8192"] = {"us_per_block": us, "gbs": b / us / 1e3, "frac_hbm": b / us / 1e3 / hbm,
                                          "bytes_per_block": b, "launches_per_block": 2}
    del L

    # fused Q4_K QKV projection (GQA 3072 -> 3072 + 1024 + 1024), 28 layers cycled
    qkv = gen_parallel([lambda t=t: synth.qkv_layer(t) for t in range(N_LAYERS)])
    LQ = [(qdq.upload_q4k(wq, synth.N_Q, N_EMBD, device=dev), qdq.upload_q4k(wk, synth.N_KV, N_EMBD, device=dev),
           qdq.upload_q4k(wv, synth.N_KV, N_EMBD, device=dev)) for wq, wk, wv in qkv]
    del qkv
    xq = torch.from_numpy(synth.activations(synth.rng_for(5, 3), 1, N_EMBD)).to(dev)
    oq, ok, ov = (torch.empty((1, n), device=dev) for n in (synth.N_Q, synth.N_KV, synth.N_KV))
    gq = capture(torch, lambda: [qdq.q4k_qkv(Wq, Wk, Wv, xq, oq, ok, ov, synth.N_Q, synth.N_KV, N_EMBD, 1)
                                 for Wq, Wk, Wv in LQ])
    for _ in range(5):
        gq.replay()
    dt = timer(gq.replay, iters)
    us = dt / (iters * N_LAYERS) * 1e6
    rows_q = synth.N_Q + 2 * synth.N_KV
    b = rows_q * (N_EMBD // 256) * 144 + N_EMBD * 4 + rows_q * 4
    rows["q4k_qkv_3072_q3072_kv1024"] = {"us_per_call": us, "gbs": b / us / 1e3, "frac_hbm": b / us / 1e3 / hbm,
                                         "bytes_per_call": b}
    del LQ

    # output projection 3072 -> 128256 (Q8_0, 418 MB: larger than L2) with the on-device argmax
    wb, xo = synth.output_projection()
    WO = qdq.upload_q8_0(wb, synth.N_VOCAB, N_EMBD, device=dev)
    del wb
    xo = torch.from_numpy(xo).to(dev)
    lo = torch.empty((1, synth.N_VOCAB), device=dev)
    io = torch.empty((1,), dtype=torch.int32, device=dev)
    vo = torch.empty((1,), device=dev)
    go = capture(torch, lambda: [qdq.q8_0_logits_argmax(WO, xo, lo, io, vo, synth.N_VOCAB, N_EMBD, 1)
                                 for _ in range(4)])
    for _ in range(3):
        go.replay()
    dt = timer(go.replay, max(5, iters // 4))
    us = dt / (max(5, iters // 4) * 4) * 1e6
    b = synth.N_VOCAB * (N_EMBD // 32) * 34 + N_EMBD * 4 + synth.N_VOCAB * 4 + 8
    rows["q8_0_logits_argmax_3072x128256"] = {"us_per_call": us, "gbs": b / us / 1e3, "frac_hbm": b / us / 1e3 / hbm,
                                              "bytes_per_call": b, "launches_per_call": 2}

    # the same projection with the on-device top-40 (k candidates read back instead of the logits)
    K = 40
    wsk = torch.empty(qdq.topk_workspace_bytes(synth.N_VOCAB, 1, K), dtype=torch.uint8, device=dev)
    ik = torch.empty((1, K), dtype=torch.int32, device=dev)
    vk = torch.empty((1, K), device=dev)
    gk = capture(torch, lambda: [qdq.q8_0_logits_topk(WO, xo, lo, wsk, ik, vk, synth.N_VOCAB, N_EMBD, 1, K)
                                 for _ in range(4)])
    for _ in range(3):
        gk.replay()
    dt = timer(gk.replay, max(5, iters // 4))
    us = dt / (max(5, iters // 4) * 4) * 1e6
    b = synth.N_VOCAB * (N_EMBD // 32) * 34 + N_EMBD * 4 + synth.N_VOCAB * 4 + 8 * K
    rows["q8_0_logits_top40_3072x128256"] = {"us_per_call": us, "gbs": b / us / 1e3, "frac_hbm": b / us / 1e3 / hbm,
                                             "bytes_per_call": b, "launches_per_call": 4}
    del WO

    # Q6_K output projection 3072 -> 128256 (323 MB, larger than L2)
    wb, xq6 = synth.q6k_output_projection()
    W6 = qdq.upload_q6k(wb, synth.N_VOCAB, N_EMBD, device=dev)
    del wb
    xq6 = torch.from_numpy(xq6).to(dev)
    y6 = torch.empty((1, synth.N_VOCAB), device=dev)
    g6 = capture(torch, lambda: [qdq.q6k_gemv(W6, xq6, y6, synth.N_VOCAB, N_EMBD, 1) for _ in range(4)])
    for _ in range(3):
        g6.replay()
    dt = timer(g6.replay, max(5, iters // 4))
    us = dt / (max(5, iters // 4) * 4) * 1e6
    b = synth.N_VOCAB * (N_EMBD // 256) * 210 + N_EMBD * 4 + synth.N_VOCAB * 4
    rows["q6k_gemv_3072x128256"] = {"us_per_call": us, "gbs": b / us / 1e3, "frac_hbm": b / us / 1e3 / hbm,
                                    "bytes_per_call": b}
    del W6

    # config 4: tensor-core batch GEMM, 8 copies of each shape cycled
    ncopy = 8
    for kind, (n_out, n_in) in ((0, (N_FF, N_EMBD)), (1, (N_EMBD, N_FF))):
        wsq = gen_parallel([lambda t=t: synth.config4_w(kind, t) for t in range(ncopy)])
        Wq = [qdq.upload_q8_0(w, n_out, n_in, device=dev) for w in wsq]
        del wsq
        for M in synth.C4_M:
            X = torch.from_numpy(synth.config4_x(kind, M)).to(dev)
            Y = torch.empty((M, n_out), device=dev)
            wsp = torch.empty(qdq.gemm_batch_workspace_bytes(M, n_out, n_in), dtype=torch.uint8, device=dev)
            gq = capture(torch, lambda: [qdq.q8_0_gemm_batch(w, X, Y, wsp, n_out, n_in, M) for w in Wq])
            for _ in range(3):
                gq.replay()
            it = max(10, iters // 2)
            dt = timer(gq.replay, it)
            us = dt / (it * ncopy) * 1e6
            b = Q8_W_BYTES + M * n_in * 4 + M * n_out * 4
            flops = 2.0 * M * n_out * n_in
            r = {"us_per_call": us, "gbs": b / us / 1e3, "tflops": flops / us / 1e6, "bytes_per_call": b,
                 "flop_per_call": flops, "frac_hbm": b / us / 1e3 / hbm,
                 "frac_bf16": flops / us / 1e6 / peaks["bf16_tflops"]}
            r["bound"] = "tensor" if M >= 256 else "hbm"
            rows["q8_0_gemm_%s_M%d" % ("3072x8192" if kind == 0 else "8192x3072", M)] = r
        del Wq

    # Q4_K batch GEMM on tensor cores (config-2/3 shapes, 8 copies cycled) and the M-token SwiGLU
    for kind, (n_out, n_in) in ((0, (N_FF, N_EMBD)), (1, (N_EMBD, N_FF))):
        wsq = gen_parallel([lambda t=t: synth.q4k_blocks(synth.rng_for(8, kind, t), n_out, n_in)
                            for t in range(ncopy)])
        Wq = [qdq.upload_q4k(w, n_out, n_in, device=dev) for w in wsq]
        del wsq
        for M in synth.C4_M:
            X = torch.from_numpy(synth.activations(synth.rng_for(8, 2 + kind, M), M, n_in)).to(dev)
            Y = torch.empty((M, n_out), device=dev)
            wsp = torch.empty(qdq.gemm_batch_workspace_bytes(M, n_out, n_in), dtype=torch.uint8, device=dev)
            gq = capture(torch, lambda: [qdq.q4k_gemm_batch(w, X, Y, wsp, n_out, n_in, M) for w in Wq])
            for _ in range(3):
                gq.replay()
            it = max(10, iters // 2)
            dt = timer(gq.replay, it)
            us = dt / (it * ncopy) * 1e6
            b = Q4_W_BYTES + M * n_in * 4 + M * n_out * 4
            flops = 2.0 * M * n_out * n_in
            rows["q4k_gemm_%s_M%d" % ("3072x8192" if kind == 0 else "8192x3072", M)] = {
                "us_per_call": us, "gbs": b / us / 1e3, "tflops": flops / us / 1e6, "bytes_per_call": b,
                "flop_per_call": flops, "frac_hbm": b / us / 1e3 / hbm,
                "frac_bf16": flops / us / 1e6 / peaks["bf16_tflops"], "bound": "tensor" if M >= 256 else "hbm"}
        if kind == 0:  # gate and up share the 3072 -> 8192 shape: pairs of the copies
            for M in synth.C4_M:
                X = torch.from_numpy(synth.activations(synth.rng_for(8, 4, M), M, n_in)).to(dev)
                mid = torch.empty((M, n_out), device=dev)
                wsp = torch.empty(qdq.q4k_swiglu_batch_workspace_bytes(M, n_out, n_in), dtype=torch.uint8,
                                  device=dev)
                pairs = [(Wq[2 * t], Wq[2 * t + 1]) for t in range(ncopy // 2)]
                gq = capture(torch, lambda: [qdq.q4k_swiglu_batch(a, c, X, mid, wsp, n_out, n_in, M)
                                             for a, c in pairs])
                for _ in range(3):
                    gq.replay()
                it = max(10, iters // 2)
                dt = timer(gq.replay, it)
                us = dt / (it * len(pairs)) * 1e6
                b = 2 * Q4_W_BYTES + M * n_in * 4 + M * n_out * 4
                flops = 4.0 * M * n_out * n_in
                rows["q4k_swiglu_batch_3072x8192_M%d" % M] = {
                    "us_per_call": us, "gbs": b / us / 1e3, "tflops": flops / us / 1e6, "bytes_per_call": b,
                    "flop_per_call": flops, "frac_hbm": b / us / 1e3 / hbm,
                    "frac_bf16": flops / us / 1e6 / peaks["bf16_tflops"], "bound": "tensor" if M >= 256 else "hbm"}
        del Wq
    rows["timeouts"] = qdq.pipeline_timeouts()
    return rows


def run_profile_case(case: str):
    """A few eager calls of one hot-path op on its full-size matrices (one set, no graph, no JSON line).

    For profilers: the weights are one matrix set (tens of MB), so a capture with many passes stays
    small; each call reads its weights cold when the profiler flushes the caches between passes.
    """
    import torch
    import synth
    import ggml_quantized_dequant_gb300 as qdq
    from ggml_quantized_dequant_gb300 import _build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    _build.build()
    qdq.load()
    dev = torch.device("cuda")
    calls = 5
    if case == "q8_0_gemv":
        W = qdq.upload_q8_0(synth.config1_up(0), N_FF, N_EMBD, device=dev)
        x = torch.from_numpy(synth.config1_x()).to(dev)
        y = torch.empty((1, N_FF), device=dev)
        fn = lambda: qdq.q8_0_gemv(W, x, y, N_FF, N_EMBD, 1)
    elif case == "q4k_gemv":
        W = qdq.upload_q4k(synth.config2_w(0), N_FF, N_EMBD, device=dev)
        x = torch.from_numpy(synth.config2_x()).to(dev)
        y = torch.empty((1, N_FF), device=dev)
        fn = lambda: qdq.q4k_gemv(W, x, y, N_FF, N_EMBD, 1)
    elif case == "q4k_ffn":
        g, u, d = synth.config3_layer(0)
        Wg, Wu = qdq.upload_q4k(g, N_FF, N_EMBD, device=dev), qdq.upload_q4k(u, N_FF, N_EMBD, device=dev)
        Wd = qdq.upload_q4k(d, N_EMBD, N_FF, device=dev)
        xh, rh = synth.config3_x_residual()
        x, r = torch.from_numpy(xh).to(dev), torch.from_numpy(rh).to(dev)
        out = torch.empty_like(r)
        mid = torch.empty((1, N_FF), device=dev)
        fn = lambda: qdq.q4k_ffn_residual(Wg, Wu, Wd, x, r, out, mid, N_EMBD, N_FF, 1)
    elif case.startswith("q8_0_gemm_M"):
        M = int(case[len("q8_0_gemm_M"):])
        W = qdq.upload_q8_0(synth.config4_w(0, 0), N_FF, N_EMBD, device=dev)
        X = torch.from_numpy(synth.config4_x(0, M)).to(dev)
        Y = torch.empty((M, N_FF), device=dev)
        ws = torch.empty(qdq.gemm_batch_workspace_bytes(M, N_FF, N_EMBD), dtype=torch.uint8, device=dev)
        fn = lambda: qdq.q8_0_gemm_batch(W, X, Y, ws, N_FF, N_EMBD, M)
    else:
        raise SystemExit("unknown --profile case %r" % case)
    for _ in range(calls):
        fn()
    torch.cuda.synchronize()
    if qdq.pipeline_timeouts() != 0:
        raise SystemExit("pipeline wait timed out")
    print("profile case %s: %d calls done" % (case, calls))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--row-steps", type=int, default=200, help="timed replays per extra row")
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the dominant kernel, if captured for this build")
    ap.add_argument("--profile", default=None, metavar="CASE",
                    help="run a few calls of one op for a profiler and exit: q8_0_gemv, q4k_gemv, q4k_ffn, "
                         "q8_0_gemm_M<M>")
    args = ap.parse_args(argv)
    if args.profile:
        return run_profile_case(args.profile)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
