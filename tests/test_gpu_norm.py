"""GPU parity of fused_add_rmsnorm_fp8_block_quant (MATE page "FlashInfer Wrapper
APIs", section Norm) against the CPU oracle, through the C ABI.

What must agree, and how:
  - residual (input + residual rounded to BF16): bit-exact;
  - normed_out: within one BF16 unit in the last place (the kernel reduces the
    sum of squares in FP32, the oracle in FP64), and equal almost everywhere;
  - out codes and block_scale: bit-exact in every block whose normed_out equals
    the oracle's, and in every block the exact 1 x 128 quantisation of the
    kernel's own normed_out (checked with torch's IEEE float32 division and its
    float8_e4m3fn cast, not with the oracle).
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_nt_gb300 as fp8g_pkg  # noqa: F401  (loaded through the fixture)

pytestmark = pytest.mark.gpu


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def make(rows, hidden, seed, mag=1.0):
    g = torch.Generator().manual_seed(seed)
    inp = (torch.randn((rows, hidden), generator=g) * mag).bfloat16()
    res = (torch.randn((rows, hidden), generator=g) * mag).bfloat16()
    w = (torch.randn((hidden,), generator=g) * 0.2 + 1.0).bfloat16()
    return inp, res, w


def run_gpu(fp8g, inp, res, w, eps):
    rows, hidden = inp.shape
    d_in, d_res, d_w = inp.cuda(), res.cuda(), w.cuda()
    out = torch.full((rows, hidden), 0x55, dtype=torch.uint8, device="cuda")
    bs = torch.full((rows, hidden // 128), -7.0, dtype=torch.float32, device="cuda")
    normed = torch.full((rows, hidden), -3.0, dtype=torch.bfloat16, device="cuda")
    fp8g.fused_add_rmsnorm_fp8_block_quant(out, bs, normed, d_in, d_res, d_w, eps=eps)
    torch.cuda.synchronize()
    return dict(residual_out=bits(d_res), normed_out=bits(normed), out=out.cpu().numpy(),
                block_scale=bs.cpu().numpy())


def quantise_like_the_definition(normed_bits):
    """1 x 128 E4M3 quantisation of given BF16 values with torch (IEEE float32
    division, float8_e4m3fn cast after clamping to the finite range)."""
    y = torch.from_numpy(f64(normed_bits).astype(np.float32))
    rows, hidden = y.shape
    blk = y.view(rows, hidden // 128, 128)
    amax = blk.abs().amax(dim=2)
    scale = amax / 448.0
    q = torch.where(amax[:, :, None] > 0, blk / scale[:, :, None], torch.zeros_like(blk))
    codes = q.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.view(rows, hidden).numpy(), scale.numpy()


def check(got, ref, label):
    assert np.array_equal(got["residual_out"], ref["residual_out"]), label
    gn, rn = f64(got["normed_out"]), f64(ref["normed_out"])
    ulp = np.abs(rn) * 2.0 ** -7 + 1e-38
    assert np.all(np.abs(gn - rn) <= ulp), label
    same = got["normed_out"] == ref["normed_out"]
    assert same.mean() > 0.999, (label, same.mean())
    rows, hidden = gn.shape
    block_same = same.reshape(rows, hidden // 128, 128).all(axis=2)
    gc = got["out"].reshape(rows, hidden // 128, 128)
    rc = ref["out"].reshape(rows, hidden // 128, 128)
    assert np.array_equal(gc[block_same], rc[block_same]), label
    assert np.array_equal(got["block_scale"][block_same], ref["block_scale"][block_same]), label
    codes, scale = quantise_like_the_definition(got["normed_out"])
    assert np.array_equal(got["out"], codes), label
    assert np.array_equal(got["block_scale"], scale), label


@pytest.mark.parametrize("rows,hidden,eps,mag", [
    (1, 128, 1e-6, 1.0), (3, 384, 1e-5, 1.0), (257, 1024, 1e-6, 30.0),
    (64, 7168, 1e-6, 1.0), (5, 2048, 1e-6, 1e-3), (2, 65536, 1e-6, 1.0)])
def test_full_parity(fp8g, oracle_mod, rows, hidden, eps, mag):
    inp, res, w = make(rows, hidden, seed=rows * 31 + hidden, mag=mag)
    got = run_gpu(fp8g, inp, res, w, eps)
    ref = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bits(inp), bits(res), bits(w), eps)
    check(got, ref, (rows, hidden, eps, mag))


def test_norm_workload_4096x7168_sampled_rows(fp8g, oracle_mod):
    rows, hidden = 4096, 7168
    inp, res, w = make(rows, hidden, seed=2024)
    got = run_gpu(fp8g, inp, res, w, 1e-6)
    g = torch.Generator().manual_seed(7)
    pick = torch.cat([torch.tensor([0, rows - 1]), torch.randint(1, rows - 1, (62,), generator=g)])
    ref = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bits(inp[pick]), bits(res[pick]), bits(w),
                                                       1e-6)
    sub = {k: v[pick.numpy()] for k, v in got.items()}
    check(sub, ref, "4096x7168 sampled")
    codes, scale = quantise_like_the_definition(got["normed_out"])
    assert np.array_equal(got["out"], codes)
    assert np.array_equal(got["block_scale"], scale)


def test_zero_blocks_and_rows(fp8g, oracle_mod):
    inp, res, w = make(4, 512, seed=5)
    res[1] = -inp[1]           # a whole row sums to zero: normed 0, scales 0, codes 0
    res[2, 256:384] = -inp[2, 256:384]  # one zero block inside a live row
    got = run_gpu(fp8g, inp, res, w, 1e-6)
    ref = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bits(inp), bits(res), bits(w), 1e-6)
    check(got, ref, "zeros")
    assert np.all(got["block_scale"][1] == 0) and np.all(got["out"][1] == 0)
    assert got["block_scale"][2, 2] == 0 and np.all(got["out"][2, 256:384] == 0)


def test_quantised_rows_feed_the_gemm_in_stream_order(fp8g):
    # norm -> GEMM back to back on one stream: the GEMM must read the codes and
    # scales this launch wrote (its prologue may overlap the norm kernel).
    rows, hidden, n = 512, 1024, 256
    inp, res, w = make(rows, hidden, seed=9)
    g = torch.Generator().manual_seed(10)
    b = (torch.randn((n, hidden), generator=g)).clamp(-448, 448).to(torch.float8_e4m3fn).cuda()
    b_scale = torch.rand((n // 128, hidden // 128), generator=g).add(0.5).cuda()
    d_in, d_res, d_w = inp.cuda(), res.cuda(), w.cuda()
    a = torch.empty((rows, hidden), dtype=torch.uint8, device="cuda")
    a_scale = torch.empty((rows, hidden // 128), dtype=torch.float32, device="cuda")
    normed = torch.empty((rows, hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((rows, n), dtype=torch.bfloat16, device="cuda")
    a.fill_(0)
    a_scale.fill_(0)
    fp8g.fused_add_rmsnorm_fp8_block_quant(a, a_scale, normed, d_in, d_res, d_w)
    fp8g.fp8_gemm_nt_groupwise(a, b, a_scale, b_scale, out, mma_sm=1)
    torch.cuda.synchronize()
    out2 = torch.empty_like(out)
    fp8g.fp8_gemm_nt_groupwise(a.clone(), b, a_scale.clone(), b_scale, out2, mma_sm=1)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert out.float().abs().sum() > 0


def test_invalid_arguments_launch_nothing(fp8g):
    inp, res, w = make(4, 256, seed=11)
    d_in, d_res, d_w = inp.cuda(), res.cuda(), w.cuda()
    out = torch.zeros((4, 256), dtype=torch.uint8, device="cuda")
    bs = torch.zeros((4, 2), dtype=torch.float32, device="cuda")
    normed = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    lib = fp8g.load()
    rc = lib.fused_add_rmsnorm_fp8_block_quant(out.data_ptr(), bs.data_ptr(), normed.data_ptr(),
                                               d_in.data_ptr(), d_res.data_ptr(), d_w.data_ptr(),
                                               1e-6, 4, 200, None)
    assert rc == fp8g.ERR_INVALID_ARGUMENT and "hidden" in fp8g.last_error()
    torch.cuda.synchronize()
    assert torch.equal(d_res.cpu().view(torch.int16), res.view(torch.int16))
    assert not out.any() and not bs.any()
