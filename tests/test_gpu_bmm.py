"""GPU parity of bmm_fp8 (MATE page "FlashInfer Wrapper APIs", section GEMM: A (batch, m, k) @
B (batch, k, n), E4M3 or E5M2 operands, tensorwise or channelwise FP32 scales) against the CPU
oracle, through the C ABI.  Tolerance as for the GEMMs: |gpu - ref| <= 1e-2 |ref| + 2e-3 rms(ref)
(the kernel sums the whole of k in FP32 on the tensor cores, the oracle in FP64)."""
import numpy as np
import pytest
import torch

from parity import assert_close, sentinel_like

pytestmark = pytest.mark.gpu

FMT = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}
LIM = {0: 448.0, 1: 57344.0}


def operands(batch, m, n, k, a_fmt, b_fmt, channelwise, seed):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn((batch, m, k), generator=g) * 2).clamp(-LIM[a_fmt], LIM[a_fmt]).to(FMT[a_fmt])
    b = (torch.randn((batch, k, n), generator=g) * 2).clamp(-LIM[b_fmt], LIM[b_fmt]).to(FMT[b_fmt])
    if channelwise:
        sa = torch.exp2(torch.empty((batch, m, 1)).uniform_(-4, 0, generator=g))
        sb = torch.exp2(torch.empty((batch, 1, n)).uniform_(-4, 0, generator=g))
    else:
        sa = torch.tensor([0.0625], dtype=torch.float32)
        sb = torch.tensor([0.71], dtype=torch.float32)
    return a, b, sa, sb


def run(fp8g, a, b, sa, sb, out_dtype=torch.bfloat16):
    batch, m, _ = a.shape
    n = b.shape[2]
    out = sentinel_like((batch, m, n), out_dtype, "cuda")
    fp8g.bmm_fp8(a.cuda(), b.cuda(), sa.cuda(), sb.cuda(), out=out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("a_fmt,b_fmt", [(0, 0), (1, 1), (0, 1), (1, 0)])
@pytest.mark.parametrize("channelwise", [False, True])
@pytest.mark.parametrize("shape", [(1, 128, 256, 128), (2, 200, 384, 640), (3, 1, 128, 256),
                                   (1, 300, 512, 1024)])
def test_parity(fp8g, oracle_mod, a_fmt, b_fmt, channelwise, shape):
    batch, m, n, k = shape
    a, b, sa, sb = operands(batch, m, n, k, a_fmt, b_fmt, channelwise, seed=sum(shape) + a_fmt)
    out = run(fp8g, a, b, sa, sb)
    ref, _ = oracle_mod.bmm_fp8(a.view(torch.uint8), b.view(torch.uint8), sa.numpy(), sb.numpy(),
                                a_fmt, b_fmt)
    got = out.float().cpu().double().numpy()
    assert_close(got.reshape(-1), ref.reshape(-1), "bmm %s %s %s" % (shape, a_fmt, b_fmt))


def test_f16_output_and_rows_past_m_are_not_written(fp8g, oracle_mod):
    # m = 200: the second 128-row tile of every batch reaches into the next
    # batch's rows of A; those rows must not be written
    a, b, sa, sb = operands(3, 200, 256, 384, 0, 0, True, seed=5)
    out = run(fp8g, a, b, sa, sb, torch.float16)
    ref, _ = oracle_mod.bmm_fp8(a.view(torch.uint8), b.view(torch.uint8), sa.numpy(), sb.numpy(),
                                out_dtype=oracle_mod.OUT_F16)
    assert_close(out.float().cpu().double().numpy().reshape(-1), ref.reshape(-1), "bmm f16")


def test_all_ones_closed_form_exact(fp8g):
    for fmt in (0, 1):
        a = torch.ones((2, 256, 512)).to(FMT[fmt])
        b = torch.ones((2, 512, 384)).to(FMT[fmt])
        out = run(fp8g, a, b, torch.tensor([0.5]), torch.tensor([0.25]))
        assert torch.all(out.float().cpu() == 512 * 0.5 * 0.25)


def test_tensorwise_equals_constant_channelwise_bit_exact(fp8g):
    a, b, _, _ = operands(2, 256, 256, 512, 1, 0, False, seed=6)
    t = run(fp8g, a, b, torch.tensor([0.375]), torch.tensor([1.5]))
    c = run(fp8g, a, b, torch.full((2, 256, 1), 0.375), torch.full((2, 1, 256), 1.5))
    assert torch.equal(t.view(torch.int16), c.view(torch.int16))


@pytest.mark.parametrize("shape", [(1, 2560, 2048, 1024), (3, 1024, 2048, 2048)])
def test_many_tiles_per_cta(fp8g, oracle_mod, shape):
    # more tiles than SMs with many K blocks each: every CTA runs several tiles
    # through both TMEM buffers, and the ring of slots wraps many times per tile
    batch, m, n, k = shape
    a, b, sa, sb = operands(batch, m, n, k, 0, 1, True, seed=11)
    out = run(fp8g, a, b, sa, sb)
    g = torch.Generator().manual_seed(12)
    for bb in range(batch):
        rows = torch.randint(0, m, (6,), generator=g)
        ref, _ = oracle_mod.bmm_fp8(a.view(torch.uint8)[bb:bb + 1, rows],
                                    b.view(torch.uint8)[bb:bb + 1], sa[bb:bb + 1, rows].numpy(),
                                    sb[bb:bb + 1].numpy(), 0, 1)
        got = out[bb, rows.cuda()].float().cpu().double().numpy()
        assert_close(got.reshape(-1), ref.reshape(-1), "bmm many tiles %s batch %d" % (shape, bb))


def test_bmm_workload_sampled(fp8g, oracle_mod):
    import workloads
    w = workloads.make("bmm_fp8_b4_4096x4096x7168")
    out = run(fp8g, w["A"], w["B"], w["A_scale"], w["B_scale"])
    g = torch.Generator().manual_seed(9)
    # the oracle on a few rows of every batch
    for bb in range(w["A"].shape[0]):
        rows = torch.randint(0, w["A"].shape[1], (4,), generator=g)
        ref, _ = oracle_mod.bmm_fp8(w["A"].view(torch.uint8)[bb:bb + 1, rows],
                                    w["B"].view(torch.uint8)[bb:bb + 1], w["A_scale"].numpy(),
                                    w["B_scale"].numpy())
        got = out[bb, rows.cuda()].float().cpu().double().numpy()
        assert_close(got.reshape(-1), ref.reshape(-1), "bmm workload batch %d" % bb)


@pytest.mark.parametrize("a_fmt,b_fmt", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("channelwise", [False, True])
@pytest.mark.parametrize("shape", [(2, 200, 208, 176), (1, 130, 80, 48), (3, 65, 400, 272),
                                   (1, 1, 16, 16), (2, 257, 528, 1040)])
def test_ragged_n_and_k_parity_and_no_write_past_the_output(fp8g, oracle_mod, a_fmt, b_fmt,
                                                            channelwise, shape):
    # n and k multiples of 16 but not of 128: the last K block's tail and the
    # columns past n read as zero; nothing past (batch, m, n) is written (the
    # output sits at the start of a larger sentinel buffer)
    batch, m, n, k = shape
    a, b, sa, sb = operands(batch, m, n, k, a_fmt, b_fmt, channelwise,
                            seed=sum(shape) + 7 * a_fmt + b_fmt)
    size = batch * m * n
    buf = sentinel_like((size + 4096,), torch.bfloat16, "cuda")
    guard = buf[size:].clone()
    out = buf[:size].view(batch, m, n)
    fp8g.bmm_fp8(a.cuda(), b.cuda(), sa.cuda(), sb.cuda(), out=out)
    torch.cuda.synchronize()
    assert torch.equal(buf[size:].view(torch.int16), guard.view(torch.int16))
    ref, _ = oracle_mod.bmm_fp8(a.view(torch.uint8), b.view(torch.uint8), sa.numpy(), sb.numpy(),
                                a_fmt, b_fmt)
    assert_close(out.float().cpu().double().numpy().reshape(-1), ref.reshape(-1),
                 "bmm ragged %s %s %s" % (shape, a_fmt, b_fmt))


@pytest.mark.parametrize("a_fmt,b_fmt", [(0, 0), (1, 0)])
def test_cta_pairs_ragged_full_parity_and_same_bits_as_one_cta(fp8g, oracle_mod, a_fmt, b_fmt):
    # enough 256 x 256 tiles for CTA pairs (each CTA 128 rows of A, one
    # 128-column half of B); m, n and k ragged; full parity, and the same bits
    # as the one-CTA kernel on the same batches (a problem too small for pairs,
    # run batch by batch)
    lib = fp8g.load()
    batch, m, n, k = 3, 777, 2000, 1040
    a, b, sa, sb = operands(batch, m, n, k, a_fmt, b_fmt, True, seed=61 + a_fmt)
    out = run(fp8g, a, b, sa, sb)
    assert lib.fp8g_testing_last_gemm_cta_pair() == 1
    ref, _ = oracle_mod.bmm_fp8(a.view(torch.uint8), b.view(torch.uint8), sa.numpy(), sb.numpy(),
                                a_fmt, b_fmt)
    assert_close(out.float().cpu().double().numpy().reshape(-1), ref.reshape(-1),
                 "bmm pairs %s %s" % (a_fmt, b_fmt))
    for bb in range(batch):
        one = run(fp8g, a[bb:bb + 1, :200], b[bb:bb + 1], sa[bb:bb + 1, :200], sb[bb:bb + 1])
        assert lib.fp8g_testing_last_gemm_cta_pair() == 0
        assert torch.equal(one.view(torch.int16)[0], out.view(torch.int16)[bb, :200])


def test_k_tail_reads_no_row_of_the_next_batch(fp8g, oracle_mod):
    # k = 176: the last K block covers k-rows 128..255 of each batch.  The rows
    # past k must read as zero, not as the next batch's first rows: plant
    # infinities (E5M2) there, so a read of them would turn batch 0 into NaN.
    batch, m, n, k = 2, 130, 272, 176
    a, b, sa, sb = operands(batch, m, n, k, 0, 1, True, seed=31)
    b8 = b.view(torch.uint8).clone()
    b8[1, :80, :] = 0x7C  # +inf in E5M2
    b = b8.view(torch.float8_e5m2)
    out = run(fp8g, a, b, sa, sb)
    ref, _ = oracle_mod.bmm_fp8(a.view(torch.uint8)[:1], b8[:1], sa[:1].numpy(), sb[:1].numpy(),
                                0, 1)
    got = out[:1].float().cpu().double().numpy()
    assert np.isfinite(got).all()
    assert_close(got.reshape(-1), ref.reshape(-1), "bmm batch 0 beside infinities in batch 1")


def test_argument_errors(fp8g):
    a, b, sa, sb = operands(1, 128, 256, 200, 0, 0, False, seed=7)
    with pytest.raises(fp8g.Fp8gError) as e:
        run(fp8g, a, b, sa, sb)
    assert e.value.status == fp8g.ERR_INVALID_ARGUMENT and "k = 200" in str(e.value)
    a, b, sa, sb = operands(1, 128, 200, 256, 0, 0, False, seed=7)
    with pytest.raises(fp8g.Fp8gError) as e:
        run(fp8g, a, b, sa, sb)
    assert e.value.status == fp8g.ERR_INVALID_ARGUMENT and "n = 200" in str(e.value)
