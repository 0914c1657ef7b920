"""Pins of the CPU oracle against what the page and the mathematics fix.

The oracle (oracle/oracle.c) is the plain definition of gemm_fp8_nt_groupwise
and its grouped/masked forms on the MATE page "FlashInfer Wrapper APIs",
section GEMM.  Here it is held against things other than itself: a hand-worked
example, an exact rational brute force, closed forms, exact invariants
(power-of-two scaling, layout equivalence, form reductions) and the
preconditions the page states.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = {0: "bf16", 1: "f16"}


def _rand_codes(shape, seed):
    """Random non-NaN E4M3 codes spanning the whole range (incl. subnormals)."""
    g = np.random.default_rng(seed)
    codes = g.integers(0, 256, size=shape, dtype=np.int64)
    codes[(codes & 0x7F) == 0x7F] = 0x38  # replace NaN codes
    return codes.astype(np.uint8)


def _rand_scales(shape, seed, lo=-6.0, hi=2.0):
    g = np.random.default_rng(seed)
    return np.exp2(g.uniform(lo, hi, size=shape)).astype(np.float32)


def _worked_inputs():
    with open(os.path.join(GOLDEN, "worked_dense_2x256x256.json")) as f:
        w = json.load(f)
    m, n, k = w["m"], w["n"], w["k"]
    a = np.zeros((m, k), np.uint8)
    for i, blocks in enumerate(w["a_block_codes"]):
        for kb, c in enumerate(blocks):
            a[i, kb * 128:(kb + 1) * 128] = int(c, 16)
    b = np.zeros((n, k), np.uint8)
    for jb, blocks in enumerate(w["b_block_codes_by_row_block"]):
        for kb, c in enumerate(blocks):
            b[jb * 128:(jb + 1) * 128, kb * 128:(kb + 1) * 128] = int(c, 16)
    sa = np.array(w["a_scale_k_major"], np.float32)
    sb = np.array(w["b_scale_k_major"], np.float32)
    want = np.repeat(np.array(w["expected_by_row_and_column_block"]), 128, axis=1)
    return a, b, sa, sb, want


@pytest.mark.parametrize("out_dtype", [0, 1])
@pytest.mark.parametrize("major", ["K", "MN"])
def test_hand_worked_example(oracle_mod, out_dtype, major):
    a, b, sa, sb, want = _worked_inputs()
    sm = oracle_mod.SCALE_K_MAJOR
    if major == "MN":
        sa, sb, sm = sa.T.copy(), sb.T.copy(), oracle_mod.SCALE_MN_MAJOR
    ref, bits = oracle_mod.gemm_nt_groupwise(a, b, sa, sb, sm, out_dtype)
    assert np.array_equal(ref, want)
    rounded, _ = oracle_mod.round_to(ref, out_dtype)
    assert np.array_equal(rounded, want)  # all four values are representable


def _check_against_exact(RA, ref, fmt, out_dtype, oracle_mod, kb):
    """Oracle FP64 value within its rounding bound of the exact value, and the
    16-bit result equal to the exactly rounded one (a mismatch is only allowed
    where the exact value sits within that bound of a rounding tie)."""
    R_exact, A_exact = RA
    mismatches = 0
    for i in range(ref.shape[0]):
        for j in range(ref.shape[1]):
            x = R_exact[i][j]
            got = Fraction(float(ref[i, j]))
            # each of the kb FP64 additions/products rounds by <= 2^-53 relative
            # to a partial sum bounded by sum |terms|
            bound = A_exact[i][j] * Fraction(kb + 1, 2 ** 52) + Fraction(1, 2 ** 1074)
            assert abs(got - x) <= bound, (i, j)
            want = exact.round_exact(x, fmt)
            gv = oracle_mod.round_to(np.array([ref[i, j]]), out_dtype)[0][0]
            ok = (gv == want) if isinstance(want, float) else (Fraction(float(gv)) == want)
            if not ok:
                mismatches += 1
                lo = exact.round_exact(x - bound, fmt)
                hi = exact.round_exact(x + bound, fmt)
                assert lo != hi, (i, j, x)  # only a near-tie may differ
    assert mismatches == 0


@pytest.mark.parametrize("out_dtype", [0, 1])
@pytest.mark.parametrize("major", ["K", "MN"])
def test_dense_matches_exact_brute_force(oracle_mod, out_dtype, major):
    m, n, k = 4, 256, 256
    a = _rand_codes((m, k), 10)
    b = _rand_codes((n, k), 11)
    sa = _rand_scales((m, k // 128), 12)
    sb = _rand_scales((n // 128, k // 128), 13)
    R = exact.dense(a, b, sa, sb, with_abs=True)
    sm = oracle_mod.SCALE_K_MAJOR
    if major == "MN":
        ref, bits = oracle_mod.gemm_nt_groupwise(a, b, sa.T.copy(), sb.T.copy(),
                                                 oracle_mod.SCALE_MN_MAJOR, out_dtype)
    else:
        ref, bits = oracle_mod.gemm_nt_groupwise(a, b, sa, sb, sm, out_dtype)
    _check_against_exact(R, ref, FMT[out_dtype], out_dtype, oracle_mod, k // 128)


def test_dense_matches_exact_brute_force_workload_values(oracle_mod):
    # The small workload's own value distribution (uniform[-1,1]*4, scales 2^[-4,2]).
    w = workloads.make("dense_128x256x256")
    a = w["a"][:3].numpy()
    sa = w["a_scale"][:3].numpy()
    R = exact.dense(a, w["b"].numpy(), sa, w["b_scale"].numpy(), with_abs=True)
    ref, bits = oracle_mod.gemm_nt_groupwise(a, w["b"], sa, w["b_scale"])
    _check_against_exact(R, ref, "bf16", 0, oracle_mod, 2)


def test_block_sums_are_exact(oracle_mod):
    # k = 128 and unit scales: R is the block sum itself, which must equal the
    # integer dot product of the codes' 2^-9 units, scaled by 2^-18, exactly.
    m, n, k = 16, 128, 128
    a = _rand_codes((m, k), 20)
    b = _rand_codes((n, k), 21)
    # include extreme rows: all +-448 and all smallest subnormals
    a[0] = 0x7E
    b[0] = 0x7E
    b[1] = 0xFE
    a[1] = 0x01
    one = np.ones((m, 1), np.float32)
    ref, _ = oracle_mod.gemm_nt_groupwise(a, b, one, np.ones((1, 1), np.float32))
    units = exact.UNITS
    P = units[a.astype(np.int64)] @ units[b.astype(np.int64)].T  # int64, exact
    assert np.array_equal(ref, P.astype(np.float64) * 2.0 ** -18)
    assert ref[0, 0] == 128 * 448.0 * 448.0 and ref[0, 1] == -128 * 448.0 * 448.0


def test_all_ones_closed_form(oracle_mod):
    # a = b = 1.0 everywhere, constant scales c1, c2: out = k * c1 * c2.
    m, n, k = 8, 256, 512
    a = np.full((m, k), 0x38, np.uint8)
    b = np.full((n, k), 0x38, np.uint8)
    c1, c2 = np.float32(0.3183099), np.float32(1.4142135)
    sa = np.full((m, k // 128), c1, np.float32)
    sb = np.full((n // 128, k // 128), c2, np.float32)
    ref, _ = oracle_mod.gemm_nt_groupwise(a, b, sa, sb)
    assert np.all(ref == k * float(c1) * float(c2))
    # per-block scales that are powers of two: sum_kb 128 * 2^(ea+eb), exact
    ea = np.array([[0, -3, 5, 1]], np.float32)
    eb = np.array([[2, 2, -1, 0], [0, 1, 0, -7]], np.float32)
    ref, _ = oracle_mod.gemm_nt_groupwise(a[:1], b, np.exp2(ea), np.exp2(eb))
    for jb in range(2):
        want = sum(128 * 2.0 ** (ea[0, t] + eb[jb, t]) for t in range(4))
        assert np.all(ref[0, jb * 128:(jb + 1) * 128] == want)


def test_power_of_two_scaling_is_exact(oracle_mod):
    m, n, k = 6, 384, 384
    a = _rand_codes((m, k), 30)
    b = _rand_codes((n, k), 31)
    sa = _rand_scales((m, 3), 32)
    sb = _rand_scales((3, 3), 33)
    ref, bits = oracle_mod.gemm_nt_groupwise(a, b, sa, sb)
    sa2 = sa.copy()
    sa2[2] *= 2
    r2, _ = oracle_mod.gemm_nt_groupwise(a, b, sa2, sb)
    assert np.array_equal(r2[2], 2 * ref[2])
    assert np.array_equal(np.delete(r2, 2, 0), np.delete(ref, 2, 0))
    sb2 = sb.copy()
    sb2[1] *= 0.5
    r3, _ = oracle_mod.gemm_nt_groupwise(a, b, sa, sb2)
    assert np.array_equal(r3[:, 128:256], 0.5 * ref[:, 128:256])
    assert np.array_equal(r3[:, :128], ref[:, :128])
    assert np.array_equal(r3[:, 256:], ref[:, 256:])


def test_zero_scales_isolate_one_k_block(oracle_mod):
    m, n, k = 4, 128, 384
    a = _rand_codes((m, k), 40)
    b = _rand_codes((n, k), 41)
    sa = _rand_scales((m, 3), 42)
    sb = _rand_scales((1, 3), 43)
    for keep in range(3):
        sa_k = np.zeros_like(sa)
        sa_k[:, keep] = sa[:, keep]
        ref, _ = oracle_mod.gemm_nt_groupwise(a, b, sa_k, sb)
        sl = slice(keep * 128, (keep + 1) * 128)
        one, _ = oracle_mod.gemm_nt_groupwise(
            a[:, sl].copy(), b[:, sl].copy(), sa[:, keep:keep + 1].copy(),
            sb[:, keep:keep + 1].copy())
        assert np.array_equal(ref, one)


def test_layout_equivalence_bit_exact(oracle_mod):
    w = workloads.dense(200, 384, 512, seed=50)
    ref_k, bits_k = oracle_mod.gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"])
    ref_mn, bits_mn = oracle_mod.gemm_nt_groupwise(
        w["a"], w["b"], w["a_scale"].t().contiguous(), w["b_scale"].t().contiguous(),
        oracle_mod.SCALE_MN_MAJOR)
    assert np.array_equal(ref_k, ref_mn) and np.array_equal(bits_k, bits_mn)


def test_rounding_of_results_uses_out_dtype(oracle_mod):
    w = workloads.dense(16, 128, 256, seed=51)
    ref, bits = oracle_mod.gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                             out_dtype=oracle_mod.OUT_F16)
    got = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(got, ref.astype(np.float16).astype(np.float64))


def test_sampled_equals_full(oracle_mod):
    w = workloads.dense(130, 256, 256, seed=52, scale_major="MN")
    ref, bits = oracle_mod.gemm_nt_groupwise(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                             oracle_mod.SCALE_MN_MAJOR, oracle_mod.OUT_F16)
    r, c = workloads.sample_positions(130, 256, 500, seed=3, extra_rows=(0, 129))
    rs, bs = oracle_mod.gemm_nt_groupwise_at(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                             r, c, oracle_mod.SCALE_MN_MAJOR,
                                             oracle_mod.OUT_F16)
    assert np.array_equal(rs, ref[r.numpy(), c.numpy()])
    assert np.array_equal(bs, bits[r.numpy(), c.numpy()])


def test_nan_input_propagates(oracle_mod):
    w = workloads.dense(2, 128, 128, seed=53)
    a = w["a"].clone()
    a[1, 5] = 0x7F
    ref, _ = oracle_mod.gemm_nt_groupwise(a, w["b"], w["a_scale"], w["b_scale"])
    assert np.all(np.isnan(ref[1])) and not np.any(np.isnan(ref[0]))


def test_empty_m(oracle_mod):
    a = np.zeros((0, 128), np.uint8)
    b = _rand_codes((128, 128), 54)
    ref, bits = oracle_mod.gemm_nt_groupwise(a, b, np.zeros((0, 1), np.float32),
                                             np.ones((1, 1), np.float32))
    assert ref.shape == (0, 128)


def test_dense_rejects_unaligned_k_and_n(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.gemm_nt_groupwise(np.zeros((4, 192), np.uint8), np.zeros((128, 192), np.uint8),
                                     np.ones((4, 1), np.float32), np.ones((1, 1), np.float32))
    with pytest.raises(ValueError):
        oracle_mod.gemm_nt_groupwise(np.zeros((4, 128), np.uint8), np.zeros((64, 128), np.uint8),
                                     np.ones((4, 1), np.float32), np.ones((1, 1), np.float32))


# ---------------------------------------------------------------- grouped form

def _small_grouped(seed=60, counts=(3, 0, 130, 128, 1), n=256, k=256):
    mi = []
    for e, c in enumerate(counts):
        if c:
            pad = -(-c // 128) * 128
            mi += [e] * c + [-1] * (pad - c)
    mi = torch.tensor(mi, dtype=torch.int32)
    return workloads.grouped(0, 0, len(counts), n, k, seed=seed, m_indices=mi)


def test_grouped_equals_per_expert_dense(oracle_mod):
    w = _small_grouped()
    ref, bits, written = oracle_mod.group_gemm_contiguous(
        w["a"], w["b"], w["a_scale"], w["b_scale"], w["m_indices"])
    mi = w["m_indices"].numpy()
    assert np.array_equal(written.all(axis=1), mi != -1)
    assert np.array_equal(written.any(axis=1), mi != -1)
    for e in range(w["num_groups"]):
        rows = np.nonzero(mi == e)[0]
        if rows.size == 0:
            continue
        r_e, b_e = oracle_mod.gemm_nt_groupwise(
            w["a"][rows], w["b"][e], w["a_scale"][rows], w["b_scale"][e])
        assert np.array_equal(ref[rows], r_e) and np.array_equal(bits[rows], b_e)
    assert np.all(ref[mi == -1] == 0)  # padding rows untouched (prefilled 0)


def test_grouped_matches_exact_brute_force(oracle_mod):
    w = _small_grouped(seed=61, counts=(2, 1), n=128, k=256)
    ref, bits, written = oracle_mod.group_gemm_contiguous(
        w["a"], w["b"], w["a_scale"], w["b_scale"], w["m_indices"])
    mi = w["m_indices"].numpy()
    for row in np.nonzero(mi != -1)[0]:
        e = mi[row]
        R = exact.dense(w["a"][row:row + 1].numpy(), w["b"][e].numpy(),
                        w["a_scale"][row:row + 1].numpy(), w["b_scale"][e].numpy(),
                        with_abs=True)
        _check_against_exact(R, ref[row:row + 1], "bf16", 0, oracle_mod, 2)


def test_grouped_sampled_equals_full(oracle_mod):
    w = _small_grouped(seed=62)
    ref, bits, written = oracle_mod.group_gemm_contiguous(
        w["a"], w["b"], w["a_scale"], w["b_scale"], w["m_indices"])
    r, c = workloads.sample_positions(w["m"], 256, 400, seed=4)
    rs, bs, ws = oracle_mod.group_gemm_contiguous_at(
        w["a"], w["b"], w["a_scale"], w["b_scale"], w["m_indices"], r, c)
    rr, cc = r.numpy(), c.numpy()
    assert np.array_equal(ws, written[rr, cc])
    assert np.array_equal(rs[ws], ref[rr, cc][ws]) and np.array_equal(bs[ws], bits[rr, cc][ws])


@pytest.mark.parametrize("bad", ["too_big", "below_minus_one", "two_experts_in_block"])
def test_grouped_rejects_precondition_violations(oracle_mod, bad):
    w = _small_grouped(seed=63, counts=(3, 130))
    mi = w["m_indices"].clone()
    if bad == "too_big":
        mi[0] = 2
    elif bad == "below_minus_one":
        mi[1] = -2
    else:
        mi[5] = 1  # block 0 holds expert 0 rows and now an expert 1 row
    with pytest.raises(ValueError, match="m_indices"):
        oracle_mod.group_gemm_contiguous(w["a"], w["b"], w["a_scale"], w["b_scale"], mi)


# ----------------------------------------------------------------- masked form

def test_masked_equals_per_group_dense(oracle_mod):
    mm = torch.tensor([0, 1, 130, 256, 300, -5], dtype=torch.int32)
    w = workloads.masked(6, 256, 256, 256, seed=70, masked_m=mm)
    ref, bits, written = oracle_mod.batch_gemm_masked(
        w["a"], w["b"], w["a_scale"], w["b_scale"], w["masked_m"])
    valid = [0, 1, 130, 256, 256, 0]  # clamped to [0, max_m]
    for g, v in enumerate(valid):
        assert written[g, :v].all() and not written[g, v:].any()
        if v == 0:
            continue
        r_g, b_g = oracle_mod.gemm_nt_groupwise(
            w["a"][g, :v], w["b"][g], w["a_scale"][g, :v], w["b_scale"][g])
        assert np.array_equal(ref[g, :v], r_g) and np.array_equal(bits[g, :v], b_g)


def test_masked_sampled_equals_full(oracle_mod):
    w = workloads.masked(3, 200, 128, 256, seed=71)
    ref, bits, written = oracle_mod.batch_gemm_masked(
        w["a"], w["b"], w["a_scale"], w["b_scale"], w["masked_m"])
    g = np.random.default_rng(5)
    gs, rs_, cs = g.integers(0, 3, 300), g.integers(0, 200, 300), g.integers(0, 128, 300)
    r, b, wr = oracle_mod.batch_gemm_masked_at(
        w["a"], w["b"], w["a_scale"], w["b_scale"], w["masked_m"], gs, rs_, cs)
    assert np.array_equal(wr, written[gs, rs_, cs])
    assert np.array_equal(r[wr], ref[gs, rs_, cs][wr]) and np.array_equal(b[wr], bits[gs, rs_, cs][wr])


def test_fp8_output_hand_worked_codes(oracle_mod):
    # FP8 output with output_scale (section GEMM): a = b = 1 (code 0x38),
    # k = 256, unit scales, so every R = 256 exactly; code = E4M3(256 / s).
    m, n, k = 2, 128, 256
    a = np.full((m, k), 0x38, np.uint8)
    b = np.full((n, k), 0x38, np.uint8)
    ref, _ = oracle_mod.gemm_nt_groupwise(a, b, np.ones((m, 2), np.float32),
                                          np.ones((1, 2), np.float32))
    assert np.all(ref == 256.0)
    # s = 1: 256 = 1.0 x 2^8 -> exponent field 15, mantissa 0 -> 0x78
    # s = 4: 64 = 2^6 -> exponent field 13 -> 0x68
    # s = 3: 85.33 lies in [64, 128) where the E4M3 quantum is 8: 10.67 quanta -> 88
    #        = 1.375 x 2^6 -> exponent field 13, mantissa 3 -> 0x6B
    # s = 0.5: 512 is past 448 -> saturates to 0x7E
    # s = -2: -128 = -(2^7) -> sign, exponent field 14 -> 0xF0
    for s, code in ((1.0, 0x78), (4.0, 0x68), (3.0, 0x6B), (0.5, 0x7E), (-2.0, 0xF0)):
        assert np.all(oracle_mod.quantize_output_e4m3(ref, s) == code), s


def test_fp8_output_is_the_encoder_of_the_scaled_result(oracle_mod):
    # Against torch: float32 results divided by a power-of-two scale (exact),
    # cast with float8_e4m3fn after clamping to the finite range.
    import torch
    g = np.random.default_rng(4)
    m, n, k = 64, 256, 384
    # values with at most two significant bits keep every result exact in FP32
    vals = np.array([0.0, 0.5, -0.5, 1.0, -1.0, 1.5, -1.5, 2.0, -2.0, 3.0, -3.0], np.float32)
    a = torch.from_numpy(vals[g.integers(0, vals.size, (m, k))]) \
        .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    b = torch.from_numpy(vals[g.integers(0, vals.size, (n, k))]) \
        .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    sa = np.exp2(g.integers(-3, 2, (m, 3))).astype(np.float32)
    sb = np.exp2(g.integers(-3, 2, (2, 3))).astype(np.float32)
    ref, _ = oracle_mod.gemm_nt_groupwise(a, b, sa, sb)
    # the products of codes and power-of-two scales are exact in FP32 here
    assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)
    for s in (0.125, 1.0, 8.0):
        want = torch.from_numpy((ref / s).astype(np.float32)).clamp(-448, 448) \
            .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(oracle_mod.quantize_output_e4m3(ref, s), want)
