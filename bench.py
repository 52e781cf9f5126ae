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
_DL = ["qdq_gemv_dl.cu", "qdq_internal.cuh"]
_TC = ["qdq_gemm_tc.cu", "qdq_internal.cuh"]
KERNEL_SOURCES = {
    "q8_0_gemv": _DL, "q4k_gemv": _DL, "q4k_ffn": _DL, "q4k_qkv": _DL, "q8_0_vocab": _DL, "q6k_gemv": _DL,
    "q8_0_gemm_M16": _TC, "q8_0_gemm_M64": _TC, "q8_0_gemm_M512": _TC,
    "q4k_gemm_M16": _TC, "q4k_gemm_M64": _TC, "q4k_gemm_M512": _TC,
    "q4k_swiglu_M16": _TC, "q4k_swiglu_M64": _TC, "q4k_swiglu_M512": _TC,
}


def kernel_sources_digest(case: str) -> str:
    """sha256 over the code of the CUDA sources of one profiled kernel, in the listed order:
    comments and layout are left out, so that a comment edit keeps the recorded counters."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ggml_quantized_dequant_gb300", "csrc")
    for name in KERNEL_SOURCES[case]:
        h.update(name.encode())
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(" ".join(src.split()).encode())
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

_ORACLE_DATA = None


def _oracle_init():
    """Pool-worker set-up: the config-1 layer-0 up and down matrices and their activations."""
    global _ORACLE_DATA
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    import synth
    _ORACLE_DATA = (synth.config1_up(0), synth.config1_down(0), synth.config1_x(),
                    synth.activations(synth.rng_for(1, 3), 1, N_FF))


def _oracle_unit(job):
    """One unit of CPU-oracle work: dequantise + float64 GEMV of `rows` rows (from row r0) of the
    up and of the down matrix.  Returns the algorithmic bytes of the unit and its seconds."""
    import oracle
    r0, rows = job
    if _ORACLE_DATA is None:
        _oracle_init()
    up, down, x_up, x_dn = _ORACLE_DATA
    t0 = time.perf_counter()
    for w, n_in, x in ((up, N_EMBD, x_up), (down, N_FF, x_dn)):
        a = r0 % (w.shape[0] - rows + 1)
        oracle.gemv(oracle.q8_0_dequant(w[a:a + rows], rows, n_in), x)
    dt = time.perf_counter() - t0
    nbytes = rows * (N_EMBD // 32 * 34 + N_FF // 32 * 34) + (N_EMBD + N_FF) * 4 + 2 * rows * 4
    return nbytes, dt


def host_facts():
    """(logical CPUs this process may use, CPU model string) of the machine."""
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return n, model


class OraclePool:
    """The CPU oracle on all host cores: a spawn-started process pool (safe beside CUDA)."""

    def __init__(self, cores: int):
        import multiprocessing as mp
        self.cores = cores
        self.pool = mp.get_context("spawn").Pool(cores, initializer=_oracle_init)
        self.pool.map(_oracle_unit, [(0, 8)] * cores)  # warm every worker (imports, matrices)

    def run(self, rows: int, first: int = 0):
        """One unit of `rows` rows on every core at once: (bytes, wall seconds)."""
        t0 = time.perf_counter()
        res = self.pool.map(_oracle_unit, [((first + i) * rows, rows) for i in range(self.cores)])
        return sum(b for b, _ in res), time.perf_counter() - t0

    def close(self):
        self.pool.terminate()
        self.pool.join()


def cpu_baseline(budget_s: float = 12.0):
    """The CPU oracle timed on one thread and on all host cores (GB/s of algorithmic bytes)."""
    cores, model = host_facts()
    _oracle_init()
    rows = 256
    # one thread: repeat the unit until about a third of the budget is spent
    nb1, t1, i = 0, 0.0, 0
    while t1 < budget_s / 3:
        b, dt = _oracle_unit((i * rows, rows))
        nb1, t1, i = nb1 + b, t1 + dt, i + 1
    one = nb1 / t1 / 1e9
    # all cores: one unit per core at once, repeated for the rest of the budget
    pool = OraclePool(cores)
    try:
        nbp, tp, j = 0, 0.0, 0
        while tp < budget_s / 2:
            b, dt = pool.run(rows, first=j * cores)
            nbp, tp, j = nbp + b, tp + dt, j + 1
    finally:
        pool.close()
    allc = nbp / tp / 1e9
    return {"value": allc, "unit": "GB/s", "cores": cores, "kind": "oracle", "cpu_model": model,
            "value_1_thread": one, "threads_1": 1,
            "sample": "CPU oracle (numpy: own fp16 decode, f32 dequant, float64 GEMV) on row samples of the "
                      "config-1 layer-0 up (3072->8192) and down (8192->3072) Q8_0 matrices: %d rows of each per "
                      "unit; one thread: %d units in %.1f s; all %d cores (%s, one process each): %d rounds of "
                      "%d units in %.1f s" % (rows, i, t1, cores, model, j, cores, tp)}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return 0
    cores, model = host_facts()
    pool = OraclePool(cores)
    try:
        # size each step so the whole --warmup + --steps run takes about a minute
        per_step_s = max(0.05, 60.0 / max(1, args.steps + args.warmup))
        b, dt = pool.run(16)
        rows = int(max(2, min(N_EMBD, 16 * per_step_s / max(dt, 1e-6))))
        for i in range(args.warmup):
            pool.run(rows, first=i * cores)
        nbytes, t_all = 0, 0.0
        for i in range(args.steps):
            b, dt = pool.run(rows, first=(args.warmup + i) * cores)
            nbytes, t_all = nbytes + b, t_all + dt
    finally:
        pool.close()
    gbs = nbytes / t_all / 1e9
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_all / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "sample_rows_per_matrix_per_core_per_step": rows, "batch": 1,
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "cpu_model": model,
                         "sample": "%d rows of the config-1 up and down matrices per core per step (CPU oracle, "
                                   "one process per core)" % rows},
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
        """Seconds for `iters` back-to-back calls of fn."""
        torch = self.torch
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(iters):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / 1e3

    def each(self, fn, iters: int):
        """Seconds of each of `iters` back-to-back calls of fn (an event pair around each)."""
        torch = self.torch
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
        torch.cuda.synchronize()
        ev[0].record()
        for i in range(iters):
            fn()
            ev[i + 1].record()
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) / 1e3 for i in range(iters)]


def pct(samples_us):
    """Median and 10th / 90th percentiles of a list of per-call microseconds."""
    a = np.asarray(samples_us, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90)),
            "samples": int(a.size)}


def roofline(bound, units_per_launch, launch_s, peak, unit, traffic, kernel, peak_source):
    """The roofline object of one kernel: algorithmic bytes (or FLOPs) per launch / its time, against the peak."""
    scale = 1e9 if unit == "GB/s" else 1e12
    achieved = units_per_launch / launch_s / scale
    return {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic, "peak_source": peak_source,
            ("bytes_per_launch" if unit == "GB/s" else "flop_per_launch"): units_per_launch}


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


def time_calls(torch, timer, fn_one, calls, iters, warm=3):
    """A CUDA graph of `calls` back-to-back calls of fn_one, replayed: mean seconds per call over
    `iters` replays, and the per-call distribution (each replay's time / calls) in microseconds."""
    g = capture(torch, lambda: [fn_one(i) for i in range(calls)])
    for _ in range(warm):
        g.replay()
    dt = timer(g.replay, iters)
    each = timer.each(g.replay, max(10, min(iters, 100)))
    return dt / (iters * calls), pct([t / calls * 1e6 for t in each])


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
    # the same graph, each replay timed alone: the per-matrix distribution
    dist = pct([t / launches_per_step * 1e6 for t in timer.each(g.replay, min(200, max(20, args.steps // 10)))])
    # the same chain as plain stream launches (no graph)
    plain_it = max(10, min(100, args.steps // 20))
    step()
    plain_us = timer(step, plain_it) / (plain_it * launches_per_step) * 1e6
    # the launch round trip: an empty kernel, then a host synchronisation, n times
    stream = torch.cuda.current_stream()
    for _ in range(20):
        qdq.noop()
        stream.synchronize()
    n_rt = 500
    t0 = time.perf_counter()
    for _ in range(n_rt):
        qdq.noop()
        stream.synchronize()
    rt_us = (time.perf_counter() - t0) / n_rt * 1e6

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
        lsf = dtf / (it * launches_per_step)
        rows["q8_0_decode_28L_fixed_point_optin"] = {
            "us_per_matrix": lsf * 1e6,
            "roofline": roofline("hbm", bytes_per_launch, lsf, peaks["hbm_gbs"], "GB/s", None,
                                 "gemv_xs_kernel<0, 0, 0> (ring kernel, block fixed point)", peaks["source"]),
            "arithmetic": "opt-in block fixed point (bound relative to each block's max |x|, not 1e-5 sum|w||x|)"}
        del gf
        rows.update(measure_rows(torch, qdq, synth, dev, timer, peaks, args))
    del W_up, W_dn

    line = {
        "metric": METRIC, "value": value_gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "layers": N_LAYERS, "shapes": "up 3072->8192, down 8192->3072",
                   "format": "GGML Q8_0", "us_per_matrix": us_per_matrix, "us_per_matrix_dist": dist,
                   "plain_launch_us_per_matrix": plain_us, "launch_roundtrip_us": rt_us,
                   "frac_of_hbm_peak": value_gbs / world / peaks["hbm_gbs"],
                   "l2": "inputs larger than L2: 56 distinct matrices, 1.50 GB, cycled every step",
                   "timing": "CUDA graph of one step (56 launches, programmatic dependent launch), "
                             "replayed; CUDA events on the replay stream; plain stream launches and one "
                             "event pair per replay measured beside it",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline("hbm", bytes_per_launch, launch_s, peaks["hbm_gbs"], "GB/s",
                             args.traffic if args.traffic is not None else recorded_traffic("q8_0_gemv"),
                             "gemv_dl_kernel<0, 0, 2> (up) + <0, 0, 1> (down): Q8_0 batch-1 GEMV, f32 arithmetic", peaks["source"]),
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


def _row(us_mean_s, dist, rl, **extra):
    r = {"us_per_call": us_mean_s * 1e6, "us_dist": dist, "roofline": rl}
    r.update(extra)
    return r


def measure_rows(torch, qdq, synth, dev, timer, peaks, args):
    """Every hot-path row on its own workload: microseconds per call (mean and the distribution
    over replays) and a roofline object for its dominant kernel."""
    rows = {}
    iters = max(20, args.row_steps)
    hbm, src = peaks["hbm_gbs"], peaks["source"]

    # config 0: 256 x 512 Q8_0 (L2-resident; microseconds only)
    wb, x0 = synth.config0()
    W0 = qdq.upload_q8_0(wb, 256, 512, device=dev)
    x0d = torch.from_numpy(x0).to(dev)
    y0 = torch.empty((1, 256), device=dev)
    ls, dist = time_calls(torch, timer, lambda i: qdq.q8_0_gemv(W0, x0d, y0, 256, 512, 1), 100, iters)
    rows["q8_0_gemv_256x512"] = {"us_per_call": ls * 1e6, "us_dist": dist, "roofline": "n/a (L2-resident)"}

    # config 2: Q4_K 3072 -> 8192, 28 copies cycled
    ws = gen_parallel([lambda t=t: synth.config2_w(t) for t in range(N_LAYERS)])
    W2 = [qdq.upload_q4k(w, N_FF, N_EMBD, device=dev) for w in ws]
    del ws
    x2 = torch.from_numpy(synth.config2_x()).to(dev)
    y2 = torch.empty((1, N_FF), device=dev)
    ls, dist = time_calls(torch, timer, lambda t: qdq.q4k_gemv(W2[t], x2, y2, N_FF, N_EMBD, 1), N_LAYERS, iters)
    b = Q4_W_BYTES + (N_EMBD + N_FF) * 4
    rows["q4k_gemv_3072x8192"] = _row(ls, dist, roofline("hbm", b, ls, hbm, "GB/s", recorded_traffic("q4k_gemv"),
                                                         "gemv_dl_kernel<1, 0, 2>", src))
    del W2

    # config 3: fused Q4_K FFN block with residual, 28 layers
    layers = gen_parallel([lambda t=t: synth.config3_layer(t) for t in range(N_LAYERS)])
    L = [(qdq.upload_q4k(g, N_FF, N_EMBD, device=dev), qdq.upload_q4k(u, N_FF, N_EMBD, device=dev),
          qdq.upload_q4k(d, N_EMBD, N_FF, device=dev)) for g, u, d in layers]
    del layers
    xh, rh = synth.config3_x_residual()
    x3, r3 = torch.from_numpy(xh).to(dev), torch.from_numpy(rh).to(dev)
    mid = torch.empty((1, N_FF), device=dev)
    ls, dist = time_calls(torch, timer,
                          lambda t: qdq.q4k_ffn_residual(L[t][0], L[t][1], L[t][2], x3, r3, r3, mid, N_EMBD, N_FF, 1),
                          N_LAYERS, iters)
    b = 3 * Q4_W_BYTES + N_EMBD * 4 + N_FF * 4 * 2 + N_EMBD * 4 * 2
    rows["q4k_ffn_residual_3072x8192"] = _row(
        ls, dist, roofline("hbm", b, ls, hbm, "GB/s", recorded_traffic("q4k_ffn"),
                           "gemv_dl_kernel<1, 1, 2> + gemv_dl_kernel<1, 2, 1> (2 launches per block)", src),
        launches_per_block=2)
    # FFN e2e: per block, one pinned H2D of x and one D2H of out, through the public call
    xp = torch.from_numpy(xh).pin_memory()
    op = torch.empty((1, N_EMBD), dtype=torch.float32).pin_memory()
    xe, oe = torch.empty_like(x3), torch.empty_like(r3)
    stream = torch.cuda.current_stream()

    def ffn_e2e(t):
        xe.copy_(xp, non_blocking=True)
        qdq.q4k_ffn_residual(L[t][0], L[t][1], L[t][2], xe, r3, oe, mid, N_EMBD, N_FF, 1)
        op.copy_(oe, non_blocking=True)
        stream.synchronize()

    for t in range(5):
        ffn_e2e(t)
    n_e = max(56, min(280, iters))
    t0 = time.perf_counter()
    for i in range(n_e):
        ffn_e2e(i % N_LAYERS)
    dte = (time.perf_counter() - t0) / n_e
    rows["q4k_ffn_residual_3072x8192"]["e2e"] = {
        "value": b / dte / 1e9, "unit": "GB/s", "us_per_block": dte * 1e6, "h2d_bytes_per_block": N_EMBD * 4,
        "d2h_bytes_per_block": N_EMBD * 4, "blocks": n_e,
        "path": "Python binding -> C ABI per block (no graph), pinned H2D of x and D2H of out, synchronised"}
    del L

    # fused Q4_K QKV projection (GQA 3072 -> 3072 + 1024 + 1024), 28 layers cycled
    qkv = gen_parallel([lambda t=t: synth.qkv_layer(t) for t in range(N_LAYERS)])
    LQ = [(qdq.upload_q4k(wq, synth.N_Q, N_EMBD, device=dev), qdq.upload_q4k(wk, synth.N_KV, N_EMBD, device=dev),
           qdq.upload_q4k(wv, synth.N_KV, N_EMBD, device=dev)) for wq, wk, wv in qkv]
    del qkv
    xq = torch.from_numpy(synth.activations(synth.rng_for(5, 3), 1, N_EMBD)).to(dev)
    oq, ok, ov = (torch.empty((1, n), device=dev) for n in (synth.N_Q, synth.N_KV, synth.N_KV))
    ls, dist = time_calls(torch, timer, lambda t: qdq.q4k_qkv(LQ[t][0], LQ[t][1], LQ[t][2], xq, oq, ok, ov, synth.N_Q,
                                                               synth.N_KV, N_EMBD, 1), N_LAYERS, iters)
    rows_q = synth.N_Q + 2 * synth.N_KV
    b = rows_q * (N_EMBD // 256) * 144 + N_EMBD * 4 + rows_q * 4
    rows["q4k_qkv_3072_q3072_kv1024"] = _row(ls, dist, roofline("hbm", b, ls, hbm, "GB/s", recorded_traffic("q4k_qkv"),
                                                                "gemv_dl_kernel<1, 3, 2>", src))
    del LQ

    # output projection 3072 -> 128256 (Q8_0, 418 MB: larger than L2) with the on-device argmax / top-40
    wb, xo = synth.output_projection()
    WO = qdq.upload_q8_0(wb, synth.N_VOCAB, N_EMBD, device=dev)
    del wb
    xo = torch.from_numpy(xo).to(dev)
    lo = torch.empty((1, synth.N_VOCAB), device=dev)
    io = torch.empty((1,), dtype=torch.int32, device=dev)
    vo = torch.empty((1,), device=dev)
    it4 = max(5, iters // 4)
    bw = synth.N_VOCAB * (N_EMBD // 32) * 34 + N_EMBD * 4 + synth.N_VOCAB * 4
    ls, dist = time_calls(torch, timer, lambda i: qdq.q8_0_gemv(WO, xo, lo, synth.N_VOCAB, N_EMBD, 1), 4, it4)
    rows["q8_0_gemv_3072x128256"] = _row(ls, dist, roofline("hbm", bw, ls, hbm, "GB/s",
                                                            recorded_traffic("q8_0_vocab"), "gemv_dl_kernel<0, 0, 2>", src))
    ls, dist = time_calls(torch, timer, lambda i: qdq.q8_0_logits_argmax(WO, xo, lo, io, vo, synth.N_VOCAB, N_EMBD, 1),
                          4, it4)
    rows["q8_0_logits_argmax_3072x128256"] = _row(
        ls, dist, roofline("hbm", bw + 8, ls, hbm, "GB/s", recorded_traffic("q8_0_vocab"),
                           "gemv_dl_kernel<0, 0, 2> + argmax_rows_kernel", src),
        launches_per_call=2)
    K = 40
    wsk = torch.empty(qdq.topk_workspace_bytes(synth.N_VOCAB, 1, K), dtype=torch.uint8, device=dev)
    ik = torch.empty((1, K), dtype=torch.int32, device=dev)
    vk = torch.empty((1, K), device=dev)
    ls, dist = time_calls(torch, timer, lambda i: qdq.q8_0_logits_topk(WO, xo, lo, wsk, ik, vk, synth.N_VOCAB, N_EMBD,
                                                                        1, K), 4, it4)
    rows["q8_0_logits_top40_3072x128256"] = _row(
        ls, dist, roofline("hbm", bw + 8 * K, ls, hbm, "GB/s", recorded_traffic("q8_0_vocab"),
                           "gemv_dl_kernel<0, 4, 2> (top-k epilogue) + topk_fold_kernel rounds", src))
    ls, dist = time_calls(torch, timer, lambda i: qdq.topk_rows(lo, synth.N_VOCAB, 1, K, wsk, ik, vk), 4, it4)
    rows["top40_128256"] = {"us_per_call": ls * 1e6, "us_dist": dist,
                            "roofline": "n/a (L2-resident logits, latency-bound warp sorts and folds)"}
    del WO

    # Q6_K output projection 3072 -> 128256 (323 MB, larger than L2)
    wb, xq6 = synth.q6k_output_projection()
    W6 = qdq.upload_q6k(wb, synth.N_VOCAB, N_EMBD, device=dev)
    del wb
    xq6 = torch.from_numpy(xq6).to(dev)
    y6 = torch.empty((1, synth.N_VOCAB), device=dev)
    ls, dist = time_calls(torch, timer, lambda i: qdq.q6k_gemv(W6, xq6, y6, synth.N_VOCAB, N_EMBD, 1), 4, it4)
    b = synth.N_VOCAB * (N_EMBD // 256) * 210 + N_EMBD * 4 + synth.N_VOCAB * 4
    rows["q6k_gemv_3072x128256"] = _row(ls, dist, roofline("hbm", b, ls, hbm, "GB/s", recorded_traffic("q6k_gemv"),
                                                           "gemv_dl_kernel<2, 0, 2>", src))
    del W6

    # config 4 and the Q4_K prefill shapes: tensor-core batch GEMMs, 8 copies of each shape cycled
    ncopy = 8
    for fmt in ("q8_0", "q4k"):
        for kind, (n_out, n_in) in ((0, (N_FF, N_EMBD)), (1, (N_EMBD, N_FF))):
            if fmt == "q8_0":
                wsq = gen_parallel([lambda t=t: synth.config4_w(kind, t) for t in range(ncopy)])
                Wq = [qdq.upload_q8_0(w, n_out, n_in, device=dev) for w in wsq]
                wbytes, f = Q8_W_BYTES, qdq.q8_0_gemm_batch
            else:
                wsq = gen_parallel([lambda t=t: synth.q4k_blocks(synth.rng_for(8, kind, t), n_out, n_in)
                                    for t in range(ncopy)])
                Wq = [qdq.upload_q4k(w, n_out, n_in, device=dev) for w in wsq]
                wbytes, f = Q4_W_BYTES, qdq.q4k_gemm_batch
            del wsq
            for M in synth.C4_M:
                X = torch.from_numpy(synth.config4_x(kind, M)).to(dev)
                Y = torch.empty((M, n_out), device=dev)
                wsp = torch.zeros(qdq.gemm_batch_workspace_bytes(M, n_out, n_in), dtype=torch.uint8, device=dev)
                ls, dist = time_calls(torch, timer, lambda t: f(Wq[t], X, Y, wsp, n_out, n_in, M), ncopy,
                                      max(10, iters // 2))
                b = wbytes + M * n_in * 4 + M * n_out * 4
                flops = 2.0 * M * n_out * n_in
                shape = "3072x8192" if kind == 0 else "8192x3072"
                kern = "gemm_tc_kernel<%d, %d, 1, *>" % (0 if fmt == "q8_0" else 1, min(256, max(16, 1 << (M - 1).bit_length())))
                # ncu traffic was captured on the 3072 -> 8192 shape; the other shape reports none
                tr = recorded_traffic("%s_gemm_M%d" % (fmt, M)) if kind == 0 else None
                if M >= 256:
                    rl = roofline("tensor", flops, ls, peaks["bf16_tflops"], "TFLOP/s", tr, kern, src)
                else:
                    rl = roofline("hbm", b, ls, hbm, "GB/s", tr, kern, src)
                rows["%s_gemm_%s_M%d" % (fmt, shape, M)] = _row(ls, dist, rl, gbs=b / ls / 1e9,
                                                               tflops=flops / ls / 1e12, bytes_per_call=b,
                                                               flop_per_call=flops)
            if fmt == "q4k" and kind == 0:  # the M-token SwiGLU: gate / up pairs of the copies
                pairs = [(Wq[2 * t], Wq[2 * t + 1]) for t in range(ncopy // 2)]
                for M in synth.C4_M:
                    X = torch.from_numpy(synth.activations(synth.rng_for(8, 4, M), M, n_in)).to(dev)
                    midb = torch.empty((M, n_out), device=dev)
                    wsp = torch.zeros(qdq.q4k_swiglu_batch_workspace_bytes(M, n_out, n_in), dtype=torch.uint8,
                                      device=dev)
                    ls, dist = time_calls(torch, timer, lambda t: qdq.q4k_swiglu_batch(
                        pairs[t][0], pairs[t][1], X, midb, wsp, n_out, n_in, M), len(pairs), max(10, iters // 2))
                    b = 2 * Q4_W_BYTES + M * n_in * 4 + M * n_out * 4
                    flops = 4.0 * M * n_out * n_in
                    kern = "gemm_tc_kernel<1, %d, 2, *>" % min(256, max(16, 1 << (M - 1).bit_length()))
                    tr = recorded_traffic("q4k_swiglu_M%d" % M)
                    rl = (roofline("tensor", flops, ls, peaks["bf16_tflops"], "TFLOP/s", tr, kern, src) if M >= 256
                          else roofline("hbm", b, ls, hbm, "GB/s", tr, kern, src))
                    rows["q4k_swiglu_batch_3072x8192_M%d" % M] = _row(ls, dist, rl, gbs=b / ls / 1e9,
                                                                     tflops=flops / ls / 1e12, bytes_per_call=b,
                                                                     flop_per_call=flops)
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
    elif case == "q4k_qkv":
        wq, wk, wv = synth.qkv_layer(0)
        Wq, Wk = qdq.upload_q4k(wq, synth.N_Q, N_EMBD, device=dev), qdq.upload_q4k(wk, synth.N_KV, N_EMBD, device=dev)
        Wv = qdq.upload_q4k(wv, synth.N_KV, N_EMBD, device=dev)
        x = torch.from_numpy(synth.activations(synth.rng_for(5, 3), 1, N_EMBD)).to(dev)
        oq, ok, ov = (torch.empty((1, n), device=dev) for n in (synth.N_Q, synth.N_KV, synth.N_KV))
        fn = lambda: qdq.q4k_qkv(Wq, Wk, Wv, x, oq, ok, ov, synth.N_Q, synth.N_KV, N_EMBD, 1)
    elif case in ("q8_0_vocab", "q6k_gemv"):
        # a 40000-row slice of the vocabulary projection (130 MB of Q8_0 / 98 MB of Q6_K): larger than
        # L2 or near it, a few hundred MB on the device at most; traffic scales with the rows
        n = 40000
        x = torch.from_numpy(synth.activations(synth.rng_for(6, 1), 1, N_EMBD)).to(dev)
        y = torch.empty((1, n), device=dev)
        if case == "q8_0_vocab":
            W = qdq.upload_q8_0(synth.q8_0_blocks(synth.rng_for(6, 0), n, N_EMBD), n, N_EMBD, device=dev)
            fn = lambda: qdq.q8_0_gemv(W, x, y, n, N_EMBD, 1)
        else:
            W = qdq.upload_q6k(synth.q6k_blocks(synth.rng_for(7, 0), n, N_EMBD), n, N_EMBD, device=dev)
            fn = lambda: qdq.q6k_gemv(W, x, y, n, N_EMBD, 1)
    elif case.startswith("q8_0_gemm_M") or case.startswith("q4k_gemm_M"):
        M = int(case.split("_M")[1])
        if case.startswith("q8_0"):
            W = qdq.upload_q8_0(synth.config4_w(0, 0), N_FF, N_EMBD, device=dev)
            f = qdq.q8_0_gemm_batch
        else:
            W = qdq.upload_q4k(synth.q4k_blocks(synth.rng_for(8, 0, 0), N_FF, N_EMBD), N_FF, N_EMBD, device=dev)
            f = qdq.q4k_gemm_batch
        X = torch.from_numpy(synth.config4_x(0, M)).to(dev)
        Y = torch.empty((M, N_FF), device=dev)
        ws = torch.zeros(qdq.gemm_batch_workspace_bytes(M, N_FF, N_EMBD), dtype=torch.uint8, device=dev)
        fn = lambda: f(W, X, Y, ws, N_FF, N_EMBD, M)
    elif case.startswith("q4k_swiglu_M"):
        M = int(case.split("_M")[1])
        Wg = qdq.upload_q4k(synth.q4k_blocks(synth.rng_for(8, 0, 0), N_FF, N_EMBD), N_FF, N_EMBD, device=dev)
        Wu = qdq.upload_q4k(synth.q4k_blocks(synth.rng_for(8, 0, 1), N_FF, N_EMBD), N_FF, N_EMBD, device=dev)
        X = torch.from_numpy(synth.activations(synth.rng_for(8, 4, M), M, N_EMBD)).to(dev)
        mid = torch.empty((M, N_FF), device=dev)
        ws = torch.zeros(qdq.q4k_swiglu_batch_workspace_bytes(M, N_FF, N_EMBD), dtype=torch.uint8, device=dev)
        fn = lambda: qdq.q4k_swiglu_batch(Wg, Wu, X, mid, ws, N_FF, N_EMBD, M)
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
                         "q4k_qkv, q8_0_vocab, q6k_gemv, q8_0_gemm_M<M>, q4k_gemm_M<M>")
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
