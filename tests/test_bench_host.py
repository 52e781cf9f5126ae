"""Host-side logic of bench.py that needs no GPU.

* whole-job throughput = units of all ranks / the slowest rank's time;
* the max-over-ranks reduction with world size 2 over gloo on 127.0.0.1;
* the nvidia-smi clock summary (median SM clock, throttle reasons);
* the peaks file is read when present, else the documented fallback.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_job_value_uses_slowest_rank():
    assert bench.job_value(100.0, 4, 2.0) == 200.0
    assert bench.job_value(5.0, 1, 0.5) == 10.0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max(1.0 + rank * 0.5)
        bench.barrier()
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 1.5, 1: 1.5}


def test_reduce_max_single_process_is_identity():
    assert bench.reduce_max(3.25) == 3.25


def test_clock_summary_parsing():
    c = bench.ClockSampler("0")
    c.lines = [
        "0, 1980, 2070, 700.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1965, 2070, 720.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2000, 2070, 710.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s["sm_mhz"] == 1980.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3


def test_clock_summary_without_samples():
    c = bench.ClockSampler("0")
    c.lines = []
    assert c.summary()["reasons"] == ["unsampled"]


def test_measured_peaks_shape():
    p = bench.measured_peaks()
    assert p["hbm_gbs"] > 1000 and p["bf16_tflops"] > 100
    assert p["source"] in ("measured", "fallback")


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2", "--impl", "reference"])


def test_algorithmic_bytes_of_the_headline():
    # GGML encodings: Q8_0 34 B per 32 weights, Q4_K 144 B per 256; plus x read and y written in f32
    assert bench.Q8_W_BYTES == 8192 * 3072 // 32 * 34 == 26_738_688
    assert bench.Q4_W_BYTES == 8192 * 3072 // 256 * 144 == 14_155_776
    assert bench.Q8_W_BYTES + bench.GEMV_IO_BYTES == 26_783_744
    assert bench.Q4_W_BYTES + bench.GEMV_IO_BYTES == 14_200_832


def test_recorded_traffic_is_keyed_to_the_kernel_sources(monkeypatch):
    # the recorded ncu bytes are reported only for the kernel sources they were captured on
    for case in bench.KERNEL_SOURCES:
        got = bench.recorded_traffic(case)
        assert got is None or got > 0
    monkeypatch.setitem(bench.KERNEL_SOURCES, "q8_0_gemv", ["qdq_gemv_xs.cu", "qdq_internal.cuh", "qdq_api.cu"])
    assert bench.recorded_traffic("q8_0_gemv") is None
