"""Pins of the oracle's bmm_fp8 (MATE page "FlashInfer Wrapper APIs", section GEMM:
A (batch, m, k) @ B (batch, k, n) of E4M3 or E5M2 codes, tensorwise or channelwise FP32
scales, BF16/FP16 out) and of its E5M2 decode table.  CPU only."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact


def test_e5m2_table_hand_worked_and_torch(oracle_mod):
    t = oracle_mod.e5m2_table()
    # 0x3C = 0.01111.00 = 1.0; 0x7B = 0.11110.11 = 1.75 * 2^15 = 57344 (largest finite);
    # 0x01 = subnormal 1/4 * 2^-14 = 2^-16; 0x80 = -0; 0xC1 = -(1.25 * 2^1) = -2.5;
    # 0x7C = +inf; 0x7D, 0xFF = NaN
    assert t[0x3C] == 1.0 and t[0x7B] == 57344.0 and t[0x01] == 2.0 ** -16
    assert t[0x80] == 0.0 and np.signbit(t[0x80]) and t[0xC1] == -2.5
    assert np.isinf(t[0x7C]) and t[0x7C] > 0 and np.isnan(t[0x7D]) and np.isnan(t[0xFF])
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e5m2).double().numpy()
    both = np.isnan(t) & np.isnan(ref)
    assert np.array_equal(t[~both], ref[~both]) and np.array_equal(np.isnan(t), np.isnan(ref))
    for c in range(256):
        v = exact.e5m2_value(c)
        if v is not None:
            assert Fraction(float(t[c])) == v


def _codes(shape, fmt, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * scale
    dt = torch.float8_e4m3fn if fmt == 0 else torch.float8_e5m2
    lim = 448.0 if fmt == 0 else 57344.0
    return x.clamp(-lim, lim).to(dt).view(torch.uint8).numpy()


@pytest.mark.parametrize("a_fmt,b_fmt", [(0, 0), (1, 1), (0, 1), (1, 0)])
@pytest.mark.parametrize("channelwise", [False, True])
@pytest.mark.parametrize("out_fmt", ["bf16", "f16"])
def test_matches_exact_rational_restatement(oracle_mod, a_fmt, b_fmt, channelwise, out_fmt):
    batch, m, n, k = 2, 3, 4, 40
    a = _codes((batch, m, k), a_fmt, 1 + a_fmt, 3.0)
    b = _codes((batch, k, n), b_fmt, 2 + b_fmt, 3.0)
    g = torch.Generator().manual_seed(3)
    if channelwise:
        sa = torch.exp2(torch.empty((batch, m, 1)).uniform_(-3, 1, generator=g)).numpy()
        sb = torch.exp2(torch.empty((batch, 1, n)).uniform_(-3, 1, generator=g)).numpy()
    else:
        sa = np.array([0.7071068], np.float32)
        sb = np.array([1.3], np.float32)
    od = oracle_mod.OUT_F16 if out_fmt == "f16" else oracle_mod.OUT_BF16
    _, bits = oracle_mod.bmm_fp8(a, b, sa, sb, a_fmt, b_fmt, od)
    want = exact.bmm(a, b, a_fmt, b_fmt, sa, sb, out_fmt)
    got = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if out_fmt == "bf16" \
        else bits.view(np.float16).astype(np.float64)
    for idx in np.ndindex(want.shape):
        assert Fraction(got[idx]) == want[idx], idx


def test_reduces_to_the_groupwise_gemm(oracle_mod):
    # E4M3, per-row a_scale and a b_scale constant on every 128-column block:
    # bmm_fp8 equals gemm_fp8_nt_groupwise on B transposed with those scales
    m, n, k = 8, 256, 384
    a = _codes((1, m, k), 0, 4)
    b = _codes((1, k, n), 0, 5)
    g = torch.Generator().manual_seed(6)
    sa = torch.exp2(torch.randint(-3, 3, (1, m, 1), generator=g).float()).numpy()
    sbb = torch.exp2(torch.randint(-3, 3, (2,), generator=g).float()).numpy()
    sb = np.repeat(sbb, 128)[None, None, :].astype(np.float32)
    _, bits = oracle_mod.bmm_fp8(a, b, sa, sb)
    bt = np.ascontiguousarray(b[0].T)
    a_scale = np.repeat(sa[0], k // 128, axis=1).astype(np.float32)
    b_scale = np.repeat(sbb[:, None], k // 128, axis=1).astype(np.float32)
    _, gbits = oracle_mod.gemm_nt_groupwise(a[0], bt, a_scale, b_scale)
    assert np.array_equal(bits[0], gbits)


def test_all_ones_closed_form_and_tensorwise_equals_channelwise(oracle_mod):
    batch, m, n, k = 2, 4, 8, 96
    for fmt, one in ((0, 0x38), (1, 0x3C)):
        a = np.full((batch, m, k), one, np.uint8)
        b = np.full((batch, k, n), one, np.uint8)
        ref, _ = oracle_mod.bmm_fp8(a, b, np.array([0.5], np.float32),
                                    np.array([0.25], np.float32), fmt, fmt)
        assert np.all(ref == k * 0.5 * 0.25)
    a = _codes((batch, m, k), 1, 7)
    b = _codes((batch, k, n), 0, 8)
    t_ref, t_bits = oracle_mod.bmm_fp8(a, b, np.array([1.5], np.float32),
                                       np.array([0.375], np.float32), 1, 0)
    c_ref, c_bits = oracle_mod.bmm_fp8(a, b, np.full((batch, m, 1), 1.5, np.float32),
                                       np.full((batch, 1, n), 0.375, np.float32), 1, 0)
    assert np.array_equal(t_bits, c_bits) and np.array_equal(t_ref, c_ref)


def test_batches_are_independent(oracle_mod):
    a = _codes((3, 5, 64), 0, 9)
    b = _codes((3, 64, 7), 1, 10)
    sa = np.array([0.25], np.float32)
    sb = np.array([2.0], np.float32)
    _, bits = oracle_mod.bmm_fp8(a, b, sa, sb, 0, 1)
    perm = [2, 0, 1]
    _, pbits = oracle_mod.bmm_fp8(a[perm], b[perm], sa, sb, 0, 1)
    assert np.array_equal(pbits, bits[perm])
