#!/usr/bin/env python
"""Throughput of the FP8 (E4M3) groupwise-scaled NT GEMM on GB300.

One step = one pass of the whole hot path over one batch of the workload.  The
default workload is the largest dense GEMM, m=16384, n=18432, k=7168 with FP16
output and K-major scales: a step is one call.  (The dense 4096 x 7168 x 2048
workload runs once with K-major and once with MN-major scales: a step is those
two calls.)

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is device-timed TFLOP/s over the K
timed steps (CUDA events on the launching stream, inputs resident in HBM,
input sets rotated so that the working set exceeds L2).  `e2e` is the same
metric through the C ABI with host buffers: every step copies its inputs from
pinned host memory and its output back.  The reference arm (`--impl
reference`) is the CPU oracle timed on the host cores on a bounded sample.

Under torchrun (N > 1) every rank runs an independent replica of the workload
(the GEMM has no exchange step); `value` is the work of all ranks divided by
the slowest rank's time.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 groupwise GEMM TFLOP/s (device-timed) and % of GB300 dense FP8 roofline"
UNIT = "TFLOP/s"
NORM_METRIC = ("fused add-RMSNorm + 1x128 FP8 quantisation GB/s (device-timed) and % of GB300 "
               "HBM roofline")
DEFAULT_WORKLOAD = "dense_16384x18432x7168"
L2_BYTES = 129 * 1024 * 1024
FP8_OVER_BF16_NOMINAL = 4.5 / 2.25  # nominal dense FP8 / BF16 tensor rate
FP8_NOMINAL_TFLOPS = 4500.0  # GB300 dense FP8 tensor rate, vendor figure (no sparsity)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    return p.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def fp8_peak_tflops(peaks, sustained=False):
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    return peaks.get(key, peaks["bf16_tflops"]) * FP8_OVER_BF16_NOMINAL


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_block_scaled_nt_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel as it is now (same source hash) and on this workload."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,utilization.gpu")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_id), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        samples = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                samples.append(dict(sm=float(parts[0]), sm_max=float(parts[1]),
                                    power=float(parts[2]),
                                    reasons=[r for r, v in zip(self.REASONS, parts[3:7])
                                             if v.lower() == "active"],
                                    util=float(parts[7])))
            except ValueError:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [s for s in samples if s["util"] > 0] or samples
        reasons = sorted({r for s in busy for r in s["reasons"]})
        return {"sm_mhz": statistics.median(s["sm"] for s in busy),
                "sm_max_mhz": max(s["sm_max"] for s in samples),
                "power_w_max": max(s["power"] for s in busy),
                "reasons": reasons, "samples": len(busy)}


def max_over_ranks(x, device=None):
    """Largest value of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput_tflops(world, flops_per_step, steps, slowest_ms, divisor=1e12):
    """Whole-job TFLOP/s (GB/s with divisor 1e9 and work in bytes): the work of
    every rank over the slowest rank's time."""
    return world * flops_per_step * steps / (slowest_ms * 1e-3) / divisor


# --------------------------------------------------------------- workloads

def metric_of(kind):
    """(metric, unit, divisor) of a workload kind: GEMMs count FLOPs, the
    HBM-bound norm + quantisation counts bytes."""
    if kind == "norm":
        return NORM_METRIC, "GB/s", 1e9
    return METRIC, UNIT, 1e12


def workload_stats(name, w):
    """Algorithmic FLOPs and bytes of one call (valid rows only)."""
    import workloads
    cfg = workloads.CONFIGS[name]
    kind = cfg["kind"]
    if kind == "moe":
        ts = w["token_selected"].cpu()
        pairs = int((ts >= 0).sum())
        live = int(torch_unique_count(ts[ts >= 0]))
        hdim, inter, t = w["hidden"], w["inter"], w["tokens"]
        flops = 2.0 * pairs * (2 * inter * hdim + hdim * inter)
        # the live experts' weights and scales, the input and the output
        bytes_ = live * (3 * inter * hdim + 4 * (3 * inter // 128) * (hdim // 128)) + 4 * t * hdim
        return flops, bytes_, "tensor"
    if kind == "bmm":
        b_, m_, n_, k_ = w["batch"], w["m"], w["n"], w["k"]
        return 2.0 * b_ * m_ * n_ * k_, b_ * (m_ * k_ + k_ * n_ + 2 * m_ * n_) + 8, "tensor"
    if kind == "norm":
        rows, hidden = w["rows"], w["hidden"]
        # read input, residual; write residual, normed_out (BF16) and the codes
        # (1 byte), plus the weight row and one FP32 scale per 128 elements
        bytes_ = rows * hidden * (2 + 2 + 2 + 2 + 1) + 2 * hidden + 4 * rows * (hidden // 128)
        return 0.0, bytes_, "hbm"
    k = w["k"]
    n = w["n"]
    kb, nb = k // 128, n // 128
    if kind == "dense":
        m = w["m"]
        out_b = 1 if "output_scale" in w else 2
        flops = 2.0 * m * n * k
        bytes_ = m * k + n * k + 4 * (m * kb + nb * kb) + out_b * m * n
        return flops, bytes_, "tensor"
    if kind == "grouped":
        mi = w["m_indices"].cpu()
        valid = int((mi != -1).sum())
        live = int(torch_unique_count(mi[mi != -1]))
        flops = 2.0 * valid * n * k
        bytes_ = live * n * k + valid * k + 2 * valid * n + 4 * (valid * kb + live * nb * kb)
        return flops, bytes_, "tensor"
    mm = w["masked_m"].cpu().clamp(0, w["max_m"])
    s = int(mm.sum())
    live = int((mm > 0).sum())
    flops = 2.0 * s * n * k
    bytes_ = live * n * k + s * k + 2 * s * n + 4 * (s * kb + live * nb * kb)
    return flops, bytes_, "hbm"


def torch_unique_count(t):
    import torch
    return torch.unique(t).numel()


def make_sets(name, device):
    """Input sets on the device, rotated step by step so that the bytes touched
    between two uses of a set exceed L2.  Returns (sets, calls_per_step)."""
    import torch
    import workloads
    cfg = workloads.CONFIGS[name]
    if cfg["kind"] == "dense":
        layouts = tuple(cfg.get("scale_layouts", ("K",)))
    else:
        layouts = (None,)
    sets = []
    per_set = 0
    for s in range(8):
        one = []
        for li, major in enumerate(layouts):
            seed = cfg["seed"] + 100 * s + li
            if cfg["kind"] == "dense":
                w = workloads.make(name, device=device, seed=seed, scale_major=major)
                odt = {"f16": torch.float16, "e4m3": torch.uint8}.get(cfg["out_dtype"],
                                                                      torch.bfloat16)
                w["out"] = torch.empty((w["m"], w["n"]), dtype=odt, device=device)
            elif cfg["kind"] == "grouped":
                w = workloads.make(name, device=device, seed=seed)
                w["out"] = torch.empty((w["m"], w["n"]), dtype=torch.bfloat16, device=device)
            elif cfg["kind"] == "moe":
                import fp8_block_scaled_nt_gb300 as fp8g
                w = workloads.make(name, device=device, seed=seed)
                w["out"] = torch.empty((w["tokens"], w["hidden"]), dtype=torch.bfloat16,
                                       device=device)
                w["workspace"] = torch.empty(fp8g.moe_workspace_size(
                    w["tokens"], w["num_experts"], w["top_k"], w["hidden"], w["inter"]),
                    dtype=torch.uint8, device=device)
            elif cfg["kind"] == "bmm":
                w = workloads.make(name, device=device, seed=seed)
                w["out"] = torch.empty((w["batch"], w["m"], w["n"]), dtype=torch.bfloat16,
                                       device=device)
            elif cfg["kind"] == "norm":
                w = workloads.make(name, device=device, seed=seed)
                rows, hidden = w["rows"], w["hidden"]
                w["out"] = torch.empty((rows, hidden), dtype=torch.uint8, device=device)
                w["block_scale"] = torch.empty((rows, hidden // 128), dtype=torch.float32,
                                               device=device)
                w["normed_out"] = torch.empty((rows, hidden), dtype=torch.bfloat16,
                                              device=device)
            else:
                w = workloads.make(name, device=device, seed=seed)
                w["out"] = torch.empty((w["num_groups"], w["max_m"], w["n"]),
                                       dtype=torch.bfloat16, device=device)
            per_set += sum(v.numel() * v.element_size() for v in w.values()
                           if torch.is_tensor(v))
            one.append(w)
        sets.append(one)
        if per_set >= 3 * L2_BYTES:
            break
    return sets, len(layouts)


def call_args(lib, name, w, stream_handle):
    """ctypes argument tuple of the C entry point for one call."""
    import workloads
    kind = workloads.CONFIGS[name]["kind"]
    p = lambda t: t.data_ptr()  # noqa: E731
    if kind == "dense":
        import torch
        od = 1 if w["out"].dtype == torch.float16 else 0
        sm = 1 if w["scale_major"] == "MN" else 0
        os_ = w.get("output_scale")
        if os_ is not None:
            od = 2  # E4M3 codes with a per-tensor output scale
        return (lib.fp8_gemm_nt_groupwise,
                (p(w["a"]), p(w["b"]), p(w["a_scale"]), p(w["b_scale"]), p(w["out"]), od,
                 p(os_) if os_ is not None else None, w["m"], w["n"], w["k"], sm, 1, 128, 128, 0,
                 stream_handle))
    if kind == "moe":
        return (lib.fused_moe_deepseek_fp8_block_scale,
                (p(w["input"]), p(w["token_selected"]), p(w["fc1"]), p(w["fc2"]), p(w["out"]),
                 p(w["fc1_scale"]), p(w["fc2_scale"]), w["tokens"], w["num_experts"],
                 w["top_k"], w["hidden"], w["inter"], p(w["workspace"]),
                 w["workspace"].numel(), stream_handle))
    if kind == "bmm":
        import torch
        fmt = lambda t: 1 if t.dtype == torch.float8_e5m2 else 0  # noqa: E731
        return (lib.bmm_fp8,
                (p(w["A"]), p(w["B"]), fmt(w["A"]), fmt(w["B"]), p(w["A_scale"]), 0,
                 p(w["B_scale"]), 0, p(w["out"]), 0, w["batch"], w["m"], w["n"], w["k"],
                 stream_handle))
    if kind == "norm":
        return (lib.fused_add_rmsnorm_fp8_block_quant,
                (p(w["out"]), p(w["block_scale"]), p(w["normed_out"]), p(w["input"]),
                 p(w["residual"]), p(w["weight"]), w["eps"], w["rows"], w["hidden"],
                 stream_handle))
    if kind == "grouped":
        return (lib.fp8_group_gemm_contiguous,
                (p(w["a"]), p(w["b"]), p(w["a_scale"]), p(w["b_scale"]), p(w["m_indices"]),
                 p(w["out"]), w["m"], w["n"], w["k"], w["num_groups"], stream_handle))
    return (lib.fp8_batch_gemm_masked,
            (p(w["a"]), p(w["b"]), p(w["a_scale"]), p(w["b_scale"]), p(w["masked_m"]),
             w["expected_m"], p(w["out"]), w["num_groups"], w["max_m"], w["n"], w["k"],
             stream_handle))


# ------------------------------------------------------------ oracle timing

def oracle_sample_rate(name, w, seconds, seed=21):
    """Time the oracle on a bounded sample of one call: output elements of a
    GEMM, rows of the norm + quantisation.  Returns (work_per_second, samples,
    seconds_taken, threads, positions, ref, written), work in FLOPs (GEMMs) or
    algorithmic bytes (norm)."""
    import numpy as np
    import oracle
    import workloads
    cfg = workloads.CONFIGS[name]
    host = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in w.items() if k != "out"}

    def run(count):
        g = np.random.default_rng(seed)
        if cfg["kind"] == "bmm":
            import torch
            r = np.sort(g.choice(host["m"], size=min(count, host["m"]), replace=False))
            fmt = lambda t: 1 if t.dtype == torch.float8_e5m2 else 0  # noqa: E731
            t0 = time.perf_counter()
            ref, _ = oracle.bmm_fp8(host["A"].view(torch.uint8)[:1, torch.as_tensor(r)],
                                    host["B"].view(torch.uint8)[:1], host["A_scale"].numpy(),
                                    host["B_scale"].numpy(), fmt(host["A"]), fmt(host["B"]))
            return time.perf_counter() - t0, r, ref[0], np.ones(r.size, bool)
        if cfg["kind"] == "moe":
            r = np.sort(g.choice(host["tokens"], size=min(count, host["tokens"]), replace=False))
            t0 = time.perf_counter()
            ref = oracle.moe_deepseek_fp8_block_scale(host["input"][r], host["token_selected"][r],
                                                      host["fc1"], host["fc2"],
                                                      host["fc1_scale"], host["fc2_scale"])
            return time.perf_counter() - t0, r, ref, np.ones(r.size, bool)
        if cfg["kind"] == "norm":
            r = np.sort(g.choice(host["rows"], size=min(count, host["rows"]), replace=False))
            t0 = time.perf_counter()
            ref = oracle.fused_add_rmsnorm_fp8_block_quant(host["input"][r], host["residual"][r],
                                                           host["weight"], host["eps"])
            return time.perf_counter() - t0, r, ref, np.ones(r.size, bool)
        if cfg["kind"] == "dense":
            r = g.integers(0, host["m"], count)
            c = g.integers(0, host["n"], count)
            sm = oracle.SCALE_MN_MAJOR if host["scale_major"] == "MN" else oracle.SCALE_K_MAJOR
            od = oracle.OUT_F16 if cfg["out_dtype"] == "f16" else oracle.OUT_BF16
            t0 = time.perf_counter()
            ref, _ = oracle.gemm_nt_groupwise_at(host["a"], host["b"], host["a_scale"],
                                                 host["b_scale"], r, c, sm, od)
            dt = time.perf_counter() - t0
            return dt, (r, c), ref, np.ones(count, bool)
        if cfg["kind"] == "grouped":
            mi = host["m_indices"].numpy()
            valid_rows = np.nonzero(mi != -1)[0]
            r = valid_rows[g.integers(0, valid_rows.size, count)]
            c = g.integers(0, host["n"], count)
            t0 = time.perf_counter()
            ref, _, wr = oracle.group_gemm_contiguous_at(host["a"], host["b"], host["a_scale"],
                                                         host["b_scale"], host["m_indices"], r, c)
            return time.perf_counter() - t0, (r, c), ref, wr
        mm = host["masked_m"].numpy().clip(0, host["max_m"])
        groups = np.nonzero(mm > 0)[0]
        gs = groups[g.integers(0, groups.size, count)]
        rs = (g.random(count) * mm[gs]).astype(np.int64)
        cs = g.integers(0, host["n"], count)
        t0 = time.perf_counter()
        ref, _, wr = oracle.batch_gemm_masked_at(host["a"], host["b"], host["a_scale"],
                                                 host["b_scale"], host["masked_m"], gs, rs, cs)
        return time.perf_counter() - t0, (gs, rs, cs), ref, wr

    # grow a probe until it takes a measurable time, then size the sample to
    # about `seconds` of oracle work
    if cfg["kind"] == "norm":
        count, limit = 4, host["rows"]
    elif cfg["kind"] == "moe":
        count, limit = 1, host["tokens"]
    elif cfg["kind"] == "bmm":
        count, limit = 1, host["m"]
    else:
        count, limit = 4096, 50_000_000
    while True:
        dt, _, _, _ = run(count)
        if dt >= min(0.5, seconds / 4) or count >= limit:
            break
        count *= 4
    count = int(max(1, min(limit, max(count, count * seconds / max(dt, 1e-6)))))
    dt, pos, ref, wr = run(count)
    if cfg["kind"] == "norm":
        _, row_bytes, _ = workload_stats(name, dict(rows=1, hidden=host["hidden"]))
        work = row_bytes * int(wr.sum())  # algorithmic bytes of the sampled rows
    elif cfg["kind"] == "bmm":
        work = 2.0 * int(wr.sum()) * host["n"] * host["k"]
    elif cfg["kind"] == "moe":
        ts = host["token_selected"][pos]
        pairs = int((np.asarray(ts) >= 0).sum())
        work = 2.0 * pairs * 3 * host["inter"] * host["hidden"]
    else:
        work = 2.0 * host["k"] * int(wr.sum())
    return work / dt, count, dt, oracle.num_threads(), pos, ref, wr


# ------------------------------------------------------------------ arms

def run_reference(args):
    """CPU oracle arm: each step is the oracle on a bounded sample of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import workloads
    metric, unit, div = metric_of(workloads.CONFIGS[args.workload]["kind"])
    w = workloads.make(args.workload, device="cpu")
    total = args.steps + args.warmup
    per_step = max(0.05, min(5.0, args.cpu_seconds / 2, 150.0 / max(total, 1)))
    # one calibration run sizes the sample so that a step takes about per_step
    rate, count, dt, threads, _, _, _ = oracle_sample_rate(args.workload, w, per_step)
    times = []
    flops = 0.0
    for i in range(total):
        r, c_, d, th, _, _, wr = oracle_sample_rate(args.workload, w, per_step, seed=100 + i)
        if i >= args.warmup:
            times.append(d)
            flops += r * d
    elapsed = sum(times)
    value = flops / elapsed / div
    kind = workloads.CONFIGS[args.workload]["kind"]
    what = {"norm": "seeded rows per step of %s (add, RMSNorm and 1x128 quantisation of each "
                    "row in FP64)",
            "moe": "seeded tokens per step of %s (the whole layer for each token: quantisation, "
                   "its experts' fc1, SwiGLU, fc2 and the sum, in FP64)",
            "bmm": "seeded rows of batch 0 per step of %s (each row's full FP64 products and "
                   "scales)"}.get(kind, "seeded output elements per step of %s (each the full "
                                        "k-long FP64 dot product and scale promotion)")
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * elapsed / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload},
        "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle",
                         "sample": "%d " % count + what % args.workload},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import fp8_block_scaled_nt_gb300 as fp8g
    from fp8_block_scaled_nt_gb300 import _build

    rank, world, local_rank = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    _build.build()
    lib = fp8g.load()
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    kind = workload_kind(args.workload)
    metric, unit_v, div = metric_of(kind)
    sets, calls_per_step = make_sets(args.workload, dev)
    flops_call, bytes_call, bound = workload_stats(args.workload, sets[0][0])
    # the unit of `value`: FLOPs for the GEMMs, algorithmic bytes for the norm
    work_call = bytes_call if kind == "norm" else flops_call
    flops_step = work_call * calls_per_step
    calls = [[call_args(lib, args.workload, w, sh) for w in one] for one in sets]

    def step(i):
        for fn, a in calls[i % len(calls)]:
            rc = fn(*a)
            if rc != 0:
                raise fp8g.Fp8gError(rc, fn.__name__, fp8g.last_error())

    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else str(local_rank)
    sampler = ClockSampler(gpu_id)
    # settle clocks (untimed, >= 1 s of back-to-back steps), then warm up
    t_end = time.time() + 1.0
    i = 0
    while time.time() < t_end:
        step(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize(dev)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    fp8g.get_device_status(clear=True)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    region_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop()
    status = fp8g.get_device_status(clear=True)
    if status:
        raise RuntimeError("device status %#x after the timed region" % status)

    region_ms = max_over_ranks(region_ms, dev)

    # End to end through the C ABI with host buffers: every step copies the
    # inputs of every call from pinned host memory, runs the calls and copies
    # the outputs back into pinned host memory.  Steps are pipelined over two
    # device buffer sets, as a caller streaming batches would: the upload of
    # step i+1 and the readback of step i-1 run on their own streams (the copy
    # engines serve both directions at once) while step i computes.
    out_keys = OUTPUT_KEYS.get(kind, ("out",))
    in_keys = INPUT_KEYS.get(kind)
    if in_keys is None:
        in_keys = tuple(k for k, v in sets[0][0].items() if torch.is_tensor(v) and k != "out")
    host_in = [{k: w[k].cpu().pin_memory() for k in in_keys} for w in sets[0]]
    host_out = [{k: torch.empty(w[k].shape, dtype=w[k].dtype).pin_memory() for k in out_keys}
                for w in sets[0]]
    h2d = sum(hi[k].numel() * hi[k].element_size() for hi in host_in for k in in_keys)
    d2h = sum(ho[k].numel() * ho[k].element_size() for ho in host_out for k in out_keys)
    copied = set(in_keys) | set(out_keys)
    dev_sets = [sets[0], [{k: (v.clone() if k in copied else v) for k, v in w.items()}
                          for w in sets[0]]]
    dev_calls = [calls[0], [call_args(lib, args.workload, w, sh) for w in dev_sets[1]]]
    up_stream = torch.cuda.Stream(dev)
    down_stream = torch.cuda.Stream(dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    read_back = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(up_stream):
            if i >= 2:  # set b's previous step is read back (outputs may be inputs too)
                up_stream.wait_event(read_back[b])
            for w, hi in zip(dev_sets[b], host_in):
                for k in in_keys:
                    w[k].copy_(hi[k], non_blocking=True)
            uploaded[b].record(up_stream)
        stream.wait_event(uploaded[b])
        for fn, a in dev_calls[b]:
            rc = fn(*a)
            if rc != 0:
                raise fp8g.Fp8gError(rc, fn.__name__, fp8g.last_error())
        computed[b].record(stream)
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(computed[b])
            for w, ho in zip(dev_sets[b], host_out):
                for k in out_keys:
                    ho[k].copy_(w[k], non_blocking=True)
            read_back[b].record(down_stream)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(down_stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    e2e_value = throughput_tflops(world, flops_step, e2e_steps, max_over_ranks(e2e_ms, dev), div)
    value = throughput_tflops(world, flops_step, args.steps, region_ms, div)
    # our kernels per call: the MoE layer launches route, quantise, fc1, SwiGLU,
    # fc2 and combine
    launches = args.steps * calls_per_step * (6 if kind == "moe" else 1)
    # the roofline is per call of the entry point (for the MoE layer: all six
    # kernels of one call)
    avg_launch_s = region_ms * 1e-3 / (args.steps * calls_per_step)
    peaks, peaks_src = load_peaks()
    kernel_name = {"dense": "gemm_kernel<dense>", "grouped": "gemm_kernel<grouped>",
                   "masked": "gemm_kernel<masked>",
                   "norm": "fused_add_rmsnorm_quant_ring_kernel", "bmm": "bmm_kernel",
                   "moe": "moe layer (route, quantise, 2 x gemm_kernel<grouped>, SwiGLU, "
                          "combine)"}[kind]
    if bound == "tensor":
        achieved = flops_call / avg_launch_s / 1e12
        peak = fp8_peak_tflops(peaks)
        unit = "TFLOP/s"
    else:
        achieved = bytes_call / avg_launch_s / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": dram_traffic(kernel_name, args.workload),
                "peak_source": "%s (%s)" % (peaks_src, "bf16 burst x 2 nominal fp8/bf16 ratio"
                                            if bound == "tensor" else "hbm copy"),
                "kernel": kernel_name, "algorithmic_flops_per_launch": flops_call,
                "algorithmic_bytes_per_launch": bytes_call,
                "avg_launch_us": avg_launch_s * 1e6}
    if bound == "tensor":
        # the same achieved rate against the other two FP8 denominators: the
        # measured bf16 rate sustained under the power cap (x 2), and the
        # vendor's nominal dense FP8 figure
        sus = fp8_peak_tflops(peaks, sustained=True)
        roofline["frac_of_sustained"] = {"peak": sus, "frac": achieved / sus,
                                         "source": "%s bf16 sustained x 2" % peaks_src}
        roofline["frac_of_nominal"] = {"peak": FP8_NOMINAL_TFLOPS,
                                       "frac": achieved / FP8_NOMINAL_TFLOPS,
                                       "source": "GB300 dense FP8 4.5 PFLOP/s (vendor)"}

    cpu_baseline = None
    spot = None
    if rank == 0 and not args.no_cpu_baseline:
        w0 = sets[0][0]
        # the inputs of set 0's last call: the end-to-end loop copied them from
        # these host buffers (the norm updates `residual` in place on the device)
        src = dict(w0)
        src.update({k: host_in[0][k] for k in in_keys})
        rate, count, dt, threads, pos, ref, wr = oracle_sample_rate(args.workload, src,
                                                                    args.cpu_seconds)
        cpu_baseline = {"value": rate / div, "unit": unit_v, "cores": threads, "kind": "oracle",
                        "sample": "%d seeded %s of one %s call (%.1f s)"
                                  % (count, {"norm": "rows", "moe": "tokens",
                                             "bmm": "rows of batch 0"}.get(
                                      kind, "output elements"), args.workload, dt)}
        # spot check of the benchmarked kernel's output at the oracle's positions
        # (set 0 was last written by the end-to-end loop from the same inputs)
        torch.cuda.synchronize(dev)
        if kind == "norm":
            spot = norm_spot_check(w0, pos, ref)
        elif kind == "moe":
            spot = moe_spot_check(w0, pos, ref)
        elif kind == "bmm":
            got = w0["out"][0, torch.as_tensor(pos, device=w0["out"].device)].float().cpu() \
                .double().numpy()
            ref = np.asarray(ref)
            rms = float(np.sqrt(np.mean(ref ** 2)))
            ok = bool(np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 2e-3 * rms))
            spot = {"elements": int(ref.size), "rows_of_batch_0": int(len(pos)),
                    "within_tolerance": ok}
        else:
            ref = np.asarray(ref)
            rms = float(np.sqrt(np.mean(ref[wr] ** 2)))
            tol = 1e-2 * np.abs(ref[wr]) + 2e-3 * rms
            if "output_scale" in w0:
                # E4M3 codes of R / s: within one E4M3 step of the exact quotient
                s_out = float(w0["output_scale"][0])
                codes = w0["out"].cpu()[tuple(torch.as_tensor(x) for x in pos)]
                got = codes.view(torch.float8_e4m3fn).double().numpy()
                q = np.clip(ref[wr] / s_out, -448, 448)
                step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6))) - 3)
                ok = bool(np.all(np.abs(got[wr] - q) <= step + tol / s_out))
            else:
                got = w0["out"].float().cpu().double().numpy()[tuple(pos)]
                ok = bool(np.all(np.abs(got[wr] - ref[wr]) <= tol))
            spot = {"elements": int(wr.sum()), "within_tolerance": ok}

    if rank == 0:
        line = {
            "metric": metric, "value": value, "unit": unit_v, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": region_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if kind == "norm" else "fp8_e4m3",
            **({"e2e_note": "expert weights resident; each step copies the input and the "
                            "routing in and the output back"} if kind == "moe" else {}),
            "data": "synthetic",
            "config": config_block(args.workload, sets, calls_per_step, world),
            "roofline": roofline, "cpu_baseline": cpu_baseline,
            "e2e": {"value": e2e_value, "unit": unit_v, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": launches, "clocks": clocks, "spot_check": spot,
            "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# tensors copied in and out by the end-to-end leg (default: everything but
# `out` in, `out` back)
INPUT_KEYS = {"norm": ("input", "residual", "weight"),
              # the expert weights stay resident, as in serving
              "moe": ("input", "token_selected")}
OUTPUT_KEYS = {"norm": ("out", "block_scale", "normed_out", "residual"), "moe": ("out",)}


def moe_spot_check(w, tokens, ref):
    """The MoE layer's output on the oracle's tokens, within the layer's
    end-to-end bound (|gpu - ref| <= 2e-2 |ref| + 2e-2 rms(ref)); the share of
    bit-equal elements is reported, not judged (the stage-by-stage GPU tests
    pin the layer)."""
    import numpy as np
    import torch
    idx = torch.as_tensor(tokens, device=w["out"].device)
    got = w["out"][idx].float().cpu().double().numpy()
    r = (np.asarray(ref).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rms = float(np.sqrt(np.mean(r ** 2)))
    ok = bool(np.all(np.abs(got - r) <= 2e-2 * np.abs(r) + 2e-2 * rms))
    got_bits = w["out"][idx].cpu().view(torch.int16).numpy().view(np.uint16)
    exact = float(np.mean(got_bits == np.asarray(ref)))
    return {"elements": int(r.size), "tokens": int(len(tokens)), "bit_equal": exact,
            "within_tolerance": ok}


def norm_spot_check(w, rows, ref):
    """The norm + quantisation's output on the oracle's rows: the residual sum
    bit-exact, normed_out within one BF16 unit, codes and scales bit-exact in
    every block whose normed_out equals the oracle's."""
    import numpy as np
    import torch
    idx = torch.as_tensor(rows, device=w["out"].device)
    got_res = w["residual"][idx].cpu().view(torch.int16).numpy().view(np.uint16)
    got_n = w["normed_out"][idx].cpu().view(torch.int16).numpy().view(np.uint16)
    got_c = w["out"][idx].cpu().numpy()
    got_s = w["block_scale"][idx].cpu().numpy()
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)  # noqa: E731
    ok = bool(np.array_equal(got_res, ref["residual_out"]))
    gn, rn = f(got_n), f(ref["normed_out"])
    ok &= bool(np.all(np.abs(gn - rn) <= np.abs(rn) * 2.0 ** -7 + 1e-38))
    same = (got_n == ref["normed_out"]).reshape(len(rows), -1, 128).all(axis=2)
    gc = got_c.reshape(len(rows), -1, 128)
    rc = ref["out"].reshape(len(rows), -1, 128)
    ok &= bool(np.array_equal(gc[same], rc[same]))
    ok &= bool(np.array_equal(got_s[same], ref["block_scale"][same]))
    return {"elements": int(got_n.size), "rows": int(len(rows)), "within_tolerance": ok}


def workload_kind(name):
    import workloads
    return workloads.CONFIGS[name]["kind"]


def config_block(name, sets, calls_per_step, world):
    import workloads
    cfg = dict(workloads.CONFIGS[name])
    block = {"workload": name, "calls_per_step": calls_per_step,
             "l2": "inputs larger than L2: %d input sets rotated per step" % len(sets),
             "parallelism": "replicas" if world > 1 else "single"}
    block.update({k: v for k, v in cfg.items() if k not in ("kind",)})
    if cfg.get("kind") == "dense":
        block["scale_layouts"] = list(cfg.get("scale_layouts", ("K",)))
    return block


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
