"""bench.py's host-side logic on CPU: cross-rank aggregation with 2 gloo ranks,
the reference arm's JSON line, and the roofline/peak bookkeeping."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slowest
        slowest = bench.max_over_ranks(ms)
        value = bench.throughput_tflops(world, 1e12, 4, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 15.0
        # 2 ranks x 4 steps x 1e12 flop in 15 ms
        assert value == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_process_aggregation_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.throughput_tflops(1, 2e12, 10, 1000.0) == pytest.approx(20.0)


def test_fp8_peak_is_twice_the_measured_bf16_peak():
    import bench
    peaks, src = bench.load_peaks()
    assert bench.fp8_peak_tflops(peaks) == pytest.approx(2 * peaks["bf16_tflops"])


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "dense_128x256x256", "--steps", "2", "--warmup", "1",
                        "--cpu-seconds", "0.2"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_norm_workload_counts_bytes_against_hbm():
    sys.path.insert(0, ROOT)
    import bench
    metric, unit, div = bench.metric_of("norm")
    assert unit == "GB/s" and div == 1e9 and "GB/s" in metric
    flops, nbytes, bound = bench.workload_stats("norm_quant_4096x7168",
                                                dict(rows=4096, hidden=7168))
    assert flops == 0.0 and bound == "hbm"
    # 4 bytes read and 5 written per element, the weight row, one scale per 128
    assert nbytes == 4096 * 7168 * 9 + 2 * 7168 + 4 * 4096 * 56
    assert bench.throughput_tflops(1, 1e9, 5, 1000.0, 1e9) == pytest.approx(5.0)


def test_reference_arm_norm_workload_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "norm_quant_4096x7168", "--steps", "2", "--warmup", "1",
                        "--cpu-seconds", "0.5"], capture_output=True, text=True, cwd=ROOT,
                       timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and "rows" in line["cpu_baseline"]["sample"]
