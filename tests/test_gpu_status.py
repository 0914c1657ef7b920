"""Failure reporting on the GPU: a pipeline wait that runs out, and the device
status word read in the order of one stream.

Error model of the "flashmla-rs" page, section Design Notes: a status code and a
last-error message, nothing thrown, the context left usable.  The timeout is
made to happen by shortening the bound of the kernel's waits far below the
launch's running time (fp8g_testing_set_wait_limit_ns), not by breaking the
pipeline: every copy and tensor-core operation the launch starts still
completes, and the launch drains them before it frees its resources.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from parity import bits16, sentinel_like, to_device

pytestmark = pytest.mark.gpu


def _dense_single_cta(fp8g, d, m, n):
    out = sentinel_like((m, n), torch.bfloat16, "cuda")
    fp8g.fp8_gemm_nt_groupwise(d["a"], d["b"], d["a_scale"], d["b_scale"], out, mma_sm=1)
    return out


def test_wait_timeout_is_reported_and_the_next_call_is_clean(fp8g):
    lib = fp8g.load()
    # one 128 x 256 tile with 1024 K blocks: each of its waits (the storer's
    # first one lasts the whole K loop) is far longer than the 2 us limit
    m, n, k = 128, 256, 131072
    d = to_device(workloads.dense(m, n, k, seed=41))
    assert fp8g.get_device_status(clear=True) == 0
    want = bits16(_dense_single_cta(fp8g, d, m, n))
    torch.cuda.synchronize()
    assert fp8g.get_device_status(clear=True) == 0

    lib.fp8g_testing_set_wait_limit_ns(2000)
    try:
        _dense_single_cta(fp8g, d, m, n)
    finally:
        lib.fp8g_testing_set_wait_limit_ns(0)
    torch.cuda.synchronize()  # the launch returned: it drained and freed what it held
    flags = ctypes.c_uint(0)
    rc = lib.fp8g_get_device_status(ctypes.byref(flags), 1)
    assert rc == fp8g.ERR_TIMEOUT and flags.value & fp8g.DEVICE_TIMEOUT, (rc, flags.value)
    assert "timeout" in fp8g.last_error()
    assert fp8g.get_device_status(clear=True) == 0  # cleared

    # the context is usable and a normal call gives the same bits as before
    again = bits16(_dense_single_cta(fp8g, d, m, n))
    torch.cuda.synchronize()
    assert fp8g.get_device_status(clear=True) == 0
    assert np.array_equal(again, want)


def test_stream_status_reads_in_stream_order(fp8g):
    g, max_m, n, k = 2, 64, 256, 256
    w = workloads.masked(g, max_m, n, k, seed=42,
                         masked_m=torch.tensor([70, 5], dtype=torch.int32))  # 70 > max_m
    d = to_device(w)
    assert fp8g.get_device_status(clear=True) == 0
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        out = torch.empty((g, max_m, n), dtype=torch.bfloat16, device="cuda")
        fp8g.fp8_batch_gemm_masked(d["a"], d["b"], d["a_scale"], d["b_scale"], d["masked_m"],
                                   w["expected_m"], out, stream=side)
        flags = fp8g.get_stream_status(clear=True, stream=side)
    assert flags & fp8g.DEVICE_MASKED_M_CLAMPED
    assert fp8g.get_stream_status(clear=False, stream=side) == 0
    assert fp8g.get_device_status(clear=True) == 0


def test_page_wrapper_runs_large_problems_on_cta_pairs(fp8g):
    """gemm_fp8_nt_groupwise with mma_sm left out launches the CTA-pair kernel
    on a large problem; an explicit mma_sm=1 the one-CTA kernel; a tiny problem
    one CTA per tile.  Results are the same bits."""
    lib = fp8g.load()
    w = to_device(workloads.dense(4096, 2048, 512, seed=43))
    auto = fp8g.gemm_fp8_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"])
    assert lib.fp8g_testing_last_gemm_cta_pair() == 1
    single = fp8g.gemm_fp8_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"], mma_sm=1)
    assert lib.fp8g_testing_last_gemm_cta_pair() == 0
    torch.cuda.synchronize()
    assert np.array_equal(bits16(auto), bits16(single))
    t = to_device(workloads.make("dense_128x256x256"))
    fp8g.gemm_fp8_nt_groupwise(t["a"], t["b"], t["a_scale"], t["b_scale"])
    assert lib.fp8g_testing_last_gemm_cta_pair() == 0
