"""GPU parity of the dense form (gemm_fp8_nt_groupwise) against the CPU oracle.

Calls go through the C ABI (libfp8g.so via the thin binding); the oracle is fed
the very same seeded tensors.
"""
import numpy as np
import pytest
import torch

import workloads
from parity import (as_f64, assert_close, bits16, sentinel_like, to_device, written_rows)

pytestmark = pytest.mark.gpu


def _run(fp8g, w, out_dtype=torch.bfloat16, mma_sm=1, stream=None):
    d = to_device(w)
    out = sentinel_like((w["m"], w["n"]), out_dtype, "cuda")
    fp8g.fp8_gemm_nt_groupwise(d["a"], d["b"], d["a_scale"], d["b_scale"], out,
                               scale_major=w["scale_major"], mma_sm=mma_sm, stream=stream)
    torch.cuda.synchronize()
    return out


def _oracle_full(oracle_mod, w, out_dtype):
    sm = oracle_mod.SCALE_MN_MAJOR if w["scale_major"] == "MN" else oracle_mod.SCALE_K_MAJOR
    od = oracle_mod.OUT_F16 if out_dtype == torch.float16 else oracle_mod.OUT_BF16
    return oracle_mod.gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"], sm, od)


def test_small_workload_full_parity(fp8g, oracle_mod):
    w = workloads.make("dense_128x256x256")
    out = _run(fp8g, w)
    ref, bits = _oracle_full(oracle_mod, w, torch.bfloat16)
    assert written_rows(out).all()
    assert_close(as_f64(out), ref, "dense 128x256x256")
    # most elements round to the same BF16 as the exact result
    assert np.mean(bits16(out) == bits) > 0.5


@pytest.mark.parametrize("mma_sm", [1, 2])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("major", ["K", "MN"])
@pytest.mark.parametrize("mnk", [(200, 384, 384), (1, 128, 128), (7, 256, 640), (129, 640, 256),
                                 (384, 512, 1152), (520, 384, 256)])
def test_ragged_shapes_full_parity(fp8g, oracle_mod, mnk, major, out_dtype, mma_sm):
    m, n, k = mnk
    w = workloads.dense(m, n, k, seed=m * 7 + n + k, scale_major=major)
    out = _run(fp8g, w, out_dtype, mma_sm=mma_sm)
    ref, _ = _oracle_full(oracle_mod, w, out_dtype)
    assert written_rows(out).all()
    assert_close(as_f64(out), ref, "dense %s %s" % (mnk, major))


@pytest.mark.parametrize("mma_sm", [1, 2])
@pytest.mark.parametrize("out_kind", ["bf16", "e4m3"])
@pytest.mark.parametrize("m", [7, 129, 200, 263])
def test_nothing_written_past_the_last_row(fp8g, m, out_kind, mma_sm):
    # out is the first m rows of a larger buffer; the rows after it (and the
    # missing right half of the last 256-column tile, n = 384) must stay as
    # they were: the last m-block is stored partly by 8-row bulk boxes and
    # partly row by row
    n, k = 384, 256
    w = workloads.dense(m, n, k, seed=m + 5)
    d = to_device(w)
    if out_kind == "bf16":
        buf = torch.full((m + 128, n), -3.0, dtype=torch.bfloat16, device="cuda")
        fp8g.fp8_gemm_nt_groupwise(d["a"], d["b"], d["a_scale"], d["b_scale"], buf[:m],
                                   mma_sm=mma_sm)
        guard = buf[m:].view(torch.int16)
        untouched = torch.full_like(guard, int(torch.tensor(-3.0).bfloat16().view(torch.int16)))
    else:
        buf = torch.full((m + 128, n), 0x7F, dtype=torch.uint8, device="cuda")  # E4M3 NaN
        scale = torch.ones(1, dtype=torch.float32, device="cuda")
        fp8g.fp8_gemm_nt_groupwise(d["a"], d["b"], d["a_scale"], d["b_scale"], buf[:m],
                                   mma_sm=mma_sm, output_scale=scale)
        guard = buf[m:]
        untouched = torch.full_like(guard, 0x7F)
    torch.cuda.synchronize()
    assert torch.equal(guard, untouched)
    if out_kind == "e4m3":  # every row of out written (saturated codes are never NaN)
        assert not (buf[:m] == 0x7F).any()


@pytest.mark.parametrize("mma_sm", [1, 2])
def test_multi_wave_full_parity(fp8g, oracle_mod, mma_sm):
    # more tiles than SMs (or SM pairs), several K blocks, m and n tails
    w = workloads.dense(2100, 2432, 512, seed=77)
    out = _run(fp8g, w, mma_sm=mma_sm)
    ref, _ = _oracle_full(oracle_mod, w, torch.bfloat16)
    assert_close(as_f64(out), ref, "dense 2100x2432x512")


@pytest.mark.parametrize("major", ["K", "MN"])
def test_dense_4096x7168x2048_sampled(fp8g, oracle_mod, major):
    w = workloads.make("dense_4096x7168x2048", scale_major=major)
    out = _run(fp8g, w, mma_sm=0)  # the launch configuration bench.py times
    assert written_rows(out).all()
    r, c = workloads.sample_positions(w["m"], w["n"], 65536, seed=11, extra_rows=(0, w["m"] - 1))
    sm = oracle_mod.SCALE_MN_MAJOR if major == "MN" else oracle_mod.SCALE_K_MAJOR
    ref, _ = oracle_mod.gemm_nt_groupwise_at(w["a"], w["b"], w["a_scale"], w["b_scale"], r, c, sm)
    got = as_f64(out)[r.numpy(), c.numpy()]
    assert_close(got, ref, "dense 4096x7168x2048 %s" % major)


def test_dense_16384x18432x7168_f16_sampled(fp8g, oracle_mod):
    w = workloads.make("dense_16384x18432x7168", device="cuda")
    out = torch.empty((w["m"], w["n"]), dtype=torch.float16, device="cuda")
    fp8g.fp8_gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"], out, mma_sm=0)
    torch.cuda.synchronize()
    r, c = workloads.sample_positions(w["m"], w["n"], 65536, seed=12, extra_rows=(0, w["m"] - 1))
    host = {k: w[k].cpu() for k in ("a", "b", "a_scale", "b_scale")}
    ref, _ = oracle_mod.gemm_nt_groupwise_at(host["a"], host["b"], host["a_scale"],
                                             host["b_scale"], r, c, out_dtype=oracle_mod.OUT_F16)
    got = out[r.cuda(), c.cuda()].double().cpu().numpy()
    assert_close(got, ref, "dense 16384x18432x7168 f16")


def test_all_ones_closed_form_exact(fp8g):
    # a = b = 1.0, power-of-two scales: every partial is exactly 128 and every
    # product exact, so out = sum_kb 128 * sa * sb exactly.
    m, n, k = 256, 512, 512
    a = torch.full((m, k), 0x38, dtype=torch.uint8)
    b = torch.full((n, k), 0x38, dtype=torch.uint8)
    g = torch.Generator().manual_seed(5)
    ea = torch.randint(-4, 3, (m, k // 128), generator=g).float()
    eb = torch.randint(-4, 3, (n // 128, k // 128), generator=g).float()
    w = dict(a=a, b=b, a_scale=torch.exp2(ea), b_scale=torch.exp2(eb), m=m, n=n, k=k,
             scale_major="K")
    out = _run(fp8g, w)
    want = (128.0 * torch.exp2(ea)[:, None, :] * torch.exp2(eb).repeat_interleave(128, 0)[None]).sum(-1)
    assert torch.equal(out.float().cpu(), want.to(torch.bfloat16).float())


def test_power_of_two_scaling_doubles_exactly(fp8g):
    w = workloads.dense(300, 512, 768, seed=90)
    base = _run(fp8g, w)
    w2 = dict(w)
    w2["a_scale"] = w["a_scale"].clone()
    w2["a_scale"][17] *= 2.0
    w2["b_scale"] = w["b_scale"].clone()
    w2["b_scale"][2] *= 0.5
    out = _run(fp8g, w2)
    b0, b1 = base.float().cpu(), out.float().cpu()
    expect = b0.clone()
    expect[17] *= 2.0
    expect[:, 256:384] *= 0.5
    assert torch.equal(b1, expect)


def test_layout_equivalence_bit_exact(fp8g):
    wk = workloads.dense(520, 768, 1024, seed=91, scale_major="K")
    wm = workloads.dense(520, 768, 1024, seed=91, scale_major="MN")
    assert np.array_equal(bits16(_run(fp8g, wk)), bits16(_run(fp8g, wm)))


@pytest.mark.parametrize("major", ["K", "MN"])
def test_scalar_b_scale_is_the_constant_block_grid(fp8g, major):
    # the page's b_scale may be a scalar (only a non-scalar tensor must be
    # contiguous): the same result, bit for bit, as that value on every block
    w = workloads.dense(300, 640, 768, seed=93, scale_major=major)
    d = to_device(w)
    s = torch.tensor([0.03125], dtype=torch.float32, device="cuda")
    grid = torch.full_like(d["b_scale"], 0.03125)
    out1 = fp8g.gemm_fp8_nt_groupwise(d["a"], d["b"], d["a_scale"], s, scale_major_mode=major)
    out2 = fp8g.gemm_fp8_nt_groupwise(d["a"], d["b"], d["a_scale"], grid, scale_major_mode=major)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert out1.float().abs().sum() > 0


@pytest.mark.parametrize("mma_sm", [0, 2])
@pytest.mark.parametrize("mnk", [(333, 640, 512), (4096, 2048, 1024)])
def test_mma_sm_hint_does_not_change_results(fp8g, mma_sm, mnk):
    w = workloads.dense(*mnk, seed=92)
    assert np.array_equal(bits16(_run(fp8g, w, mma_sm=1)), bits16(_run(fp8g, w, mma_sm=mma_sm)))


def test_cta_pair_all_ones_and_doubling_exact(fp8g):
    m, n, k = 512, 512, 384
    a = torch.full((m, k), 0x38, dtype=torch.uint8)
    b = torch.full((n, k), 0x38, dtype=torch.uint8)
    g = torch.Generator().manual_seed(6)
    ea = torch.randint(-4, 3, (m, k // 128), generator=g).float()
    eb = torch.randint(-4, 3, (n // 128, k // 128), generator=g).float()
    w = dict(a=a, b=b, a_scale=torch.exp2(ea), b_scale=torch.exp2(eb), m=m, n=n, k=k,
             scale_major="K")
    out = _run(fp8g, w, mma_sm=2)
    want = (128.0 * torch.exp2(ea)[:, None, :] * torch.exp2(eb).repeat_interleave(128, 0)[None]).sum(-1)
    assert torch.equal(out.float().cpu(), want.to(torch.bfloat16).float())
    w2 = dict(w, a_scale=w["a_scale"].clone())
    w2["a_scale"][300] *= 2.0  # a row of the odd CTA of a pair
    out2 = _run(fp8g, w2, mma_sm=2)
    expect = out.float().cpu().clone()
    expect[300] *= 2.0
    assert torch.equal(out2.float().cpu(), expect)


def test_deterministic_and_side_stream(fp8g):
    w = workloads.dense(640, 1024, 768, seed=93)
    first = bits16(_run(fp8g, w))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        second = _run(fp8g, w, stream=s)
    s.synchronize()
    assert np.array_equal(first, bits16(second))


def test_back_to_back_launches_keep_stream_order(fp8g):
    # Each launch may start its prologue while the previous kernel on the stream
    # is finishing; it must still read and write global memory only after it.
    w1 = to_device(workloads.dense(640, 1024, 768, seed=96))
    w2 = to_device(workloads.dense(640, 1024, 768, seed=97))
    alone = sentinel_like((640, 1024), torch.bfloat16, "cuda")
    fp8g.fp8_gemm_nt_groupwise(w2["a"], w2["b"], w2["a_scale"], w2["b_scale"], alone, mma_sm=2)
    torch.cuda.synchronize()
    out = sentinel_like((640, 1024), torch.bfloat16, "cuda")
    for _ in range(3):
        for w in (w1, w2):  # both write all of `out`; the second must win
            fp8g.fp8_gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"], out, mma_sm=2)
    torch.cuda.synchronize()
    assert np.array_equal(bits16(out), bits16(alone))
    # an input rewritten between two launches is read in its new state
    a = w1["a"].clone()
    out1 = sentinel_like((640, 1024), torch.bfloat16, "cuda")
    fp8g.fp8_gemm_nt_groupwise(a, w1["b"], w1["a_scale"], w1["b_scale"], out1, mma_sm=2)
    a.copy_(w2["a"])
    out2 = sentinel_like((640, 1024), torch.bfloat16, "cuda")
    fp8g.fp8_gemm_nt_groupwise(a, w2["b"], w2["a_scale"], w2["b_scale"], out2, mma_sm=2)
    torch.cuda.synchronize()
    assert np.array_equal(bits16(out2), bits16(alone))


def test_empty_m(fp8g):
    a = torch.empty((0, 256), dtype=torch.uint8, device="cuda")
    b = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_nt_groupwise(a, b, torch.empty((0, 2), device="cuda"),
                               torch.ones((1, 2), device="cuda"), out)
    torch.cuda.synchronize()


def test_page_signature_allocates_out(fp8g, oracle_mod):
    w = workloads.dense(256, 256, 256, seed=94)
    d = to_device(w)
    a8 = d["a"].view(torch.float8_e4m3fn)
    b8 = d["b"].view(torch.float8_e4m3fn)
    out = fp8g.gemm_fp8_nt_groupwise(a8, b8, d["a_scale"], d["b_scale"], out_dtype=torch.float16)
    assert out.dtype == torch.float16 and out.shape == (256, 256)
    ref, _ = oracle_mod.gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                          out_dtype=oracle_mod.OUT_F16)
    assert_close(as_f64(out), ref, "page signature")


def test_invalid_arguments_launch_nothing(fp8g):
    w = to_device(workloads.dense(128, 256, 256, seed=95))
    out = sentinel_like((128, 256), torch.bfloat16, "cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fp8_gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"], out,
                                   scale_granularity_mnk=(1, 128, 64))
    assert e.value.status == fp8g.ERR_UNSUPPORTED
    lib = fp8g.load()
    # k not a multiple of 128, straight through the C ABI
    rc = lib.fp8_gemm_nt_groupwise(w["a"].data_ptr(), w["b"].data_ptr(), w["a_scale"].data_ptr(),
                                   w["b_scale"].data_ptr(), out.data_ptr(), 0, None, 128, 256, 200,
                                   0, 1, 128, 128, 1, None)
    assert rc == fp8g.ERR_INVALID_ARGUMENT and "k = 200" in fp8g.last_error()
    # misaligned a
    rc = lib.fp8_gemm_nt_groupwise(w["a"].data_ptr() + 8, w["b"].data_ptr(),
                                   w["a_scale"].data_ptr(), w["b_scale"].data_ptr(),
                                   out.data_ptr(), 0, None, 128, 256, 256, 0, 1, 128, 128, 1, None)
    assert rc == fp8g.ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    assert not written_rows(out).any()
    assert fp8g.get_device_status() == 0


# ----------------------------------------------- FP8 (E4M3) output with output_scale

def _decode_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def _e4m3_step(q):
    """Spacing of the E4M3 grid at |q| (2^-9 in the subnormal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6)))
    return 2.0 ** (e - 3)


def _run_fp8_out(fp8g, w, s, mma_sm):
    d = to_device(w)
    os_ = torch.tensor([s], dtype=torch.float32, device="cuda")
    out = torch.full((w["m"], w["n"]), 0x7F, dtype=torch.uint8, device="cuda")  # NaN sentinel
    fp8g.fp8_gemm_nt_groupwise(d["a"], d["b"], d["a_scale"], d["b_scale"], out,
                               scale_major=w["scale_major"], mma_sm=mma_sm, output_scale=os_)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("mma_sm", [1, 2])
@pytest.mark.parametrize("mnk", [(200, 384, 384), (7, 256, 640), (520, 384, 1152), (129, 640, 256)])
def test_fp8_output_parity(fp8g, oracle_mod, mnk, mma_sm):
    m, n, k = mnk
    w = workloads.dense(m, n, k, seed=m + 3 * n + k)
    ref, _ = _oracle_full(oracle_mod, w, torch.bfloat16)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    s = float(np.float32(rms / 64))  # the bulk of |R| / s near 64, the largest values saturate
    codes = _run_fp8_out(fp8g, w, s, mma_sm)
    assert not np.any(codes == 0x7F)  # every element written, no NaN
    q = np.clip(ref / s, -448, 448)
    tol = (1e-2 * np.abs(ref) + 2e-3 * rms) / s
    assert np.all(np.abs(_decode_e4m3(codes) - q) <= _e4m3_step(q) + tol)
    want = oracle_mod.quantize_output_e4m3(ref, s)
    assert np.mean(codes == want) > 0.99


def test_fp8_output_closed_form_exact(fp8g, oracle_mod):
    # a = b = 1, power-of-two block scales and output scale: R and R / s are
    # exact in FP32, so every code is determined
    m, n, k = 256, 512, 512
    a = torch.full((m, k), 0x38, dtype=torch.uint8)
    b = torch.full((n, k), 0x38, dtype=torch.uint8)
    g = torch.Generator().manual_seed(8)
    ea = torch.randint(-5, 3, (m, k // 128), generator=g).float()
    eb = torch.randint(-5, 3, (n // 128, k // 128), generator=g).float()
    w = dict(a=a, b=b, a_scale=torch.exp2(ea), b_scale=torch.exp2(eb), m=m, n=n, k=k,
             scale_major="K")
    ref, _ = _oracle_full(oracle_mod, w, torch.bfloat16)
    for mma_sm in (1, 2):
        for s in (0.25, 1.0, 2.0):
            codes = _run_fp8_out(fp8g, w, s, mma_sm)
            assert np.array_equal(codes, oracle_mod.quantize_output_e4m3(ref, s)), (mma_sm, s)


def test_fp8_output_scale_doubling_halves_values_exactly(fp8g):
    w = workloads.dense(384, 512, 768, seed=98)
    c1 = _decode_e4m3(_run_fp8_out(fp8g, w, 0.05, 2))
    c2 = _decode_e4m3(_run_fp8_out(fp8g, w, 0.1, 2))
    normal = (np.abs(c1) >= 2.0 ** -5) & (np.abs(c1) < 448)  # away from subnormals and saturation
    assert normal.mean() > 0.5
    assert np.array_equal(c2[normal] * 2, c1[normal])


def test_fp8_output_page_signature(fp8g, oracle_mod):
    w = workloads.dense(256, 256, 512, seed=99)
    d = to_device(w)
    os_ = torch.tensor([0.02], dtype=torch.float32, device="cuda")
    out = fp8g.gemm_fp8_nt_groupwise(d["a"].view(torch.float8_e4m3fn),
                                     d["b"].view(torch.float8_e4m3fn), d["a_scale"], d["b_scale"],
                                     output_scale=os_)
    assert out.dtype == torch.float8_e4m3fn and out.shape == (256, 256)
    ref, _ = _oracle_full(oracle_mod, w, torch.bfloat16)
    q = np.clip(ref / float(os_.item()), -448, 448)
    got = out.cpu().view(torch.uint8).numpy()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    tol = (1e-2 * np.abs(ref) + 2e-3 * rms) / float(os_.item())
    assert np.all(np.abs(_decode_e4m3(got) - q) <= _e4m3_step(q) + tol)


def test_fp8_output_4096x7168x2048_sampled(fp8g, oracle_mod):
    w = workloads.make("dense_4096x7168x2048_e4m3out")
    s = float(w["output_scale"][0])
    codes = _run_fp8_out(fp8g, w, s, 0)  # the launch configuration bench.py times
    r, c = workloads.sample_positions(w["m"], w["n"], 65536, seed=13, extra_rows=(0, w["m"] - 1))
    ref, _ = oracle_mod.gemm_nt_groupwise_at(w["a"], w["b"], w["a_scale"], w["b_scale"], r, c)
    got = codes[r.numpy(), c.numpy()]
    q = np.clip(ref / s, -448, 448)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    tol = (1e-2 * np.abs(ref) + 2e-3 * rms) / s
    assert np.all(np.abs(_decode_e4m3(got) - q) <= _e4m3_step(q) + tol)
    assert np.mean(got == oracle_mod.quantize_output_e4m3(ref, s)) > 0.99


def test_fp8_output_argument_errors(fp8g):
    w = to_device(workloads.dense(128, 256, 256, seed=100))
    out8 = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):  # E4M3 out without output_scale
        fp8g.fp8_gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"], out8)
    lib = fp8g.load()
    os_ = torch.ones(1, dtype=torch.float32, device="cuda")
    rc = lib.fp8_gemm_nt_groupwise(w["a"].data_ptr(), w["b"].data_ptr(), w["a_scale"].data_ptr(),
                                   w["b_scale"].data_ptr(), out8.data_ptr(), 0, os_.data_ptr(),
                                   128, 256, 256, 0, 1, 128, 128, 1, None)
    assert rc == fp8g.ERR_INVALID_ARGUMENT and "output_scale" in fp8g.last_error()
    torch.cuda.synchronize()
    assert not out8.any()
