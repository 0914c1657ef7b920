"""Pins of the oracle's E4M3 encoder and of its fused add-RMSNorm + 1 x 128 FP8
quantisation (MATE page "FlashInfer Wrapper APIs", section Norm:
fused_add_rmsnorm_fp8_block_quant).  CPU only.

Each pin ties the oracle to something other than itself: a hand-worked example
under tests/golden/, torch's float8_e4m3fn cast and float32 -> bfloat16 cast, an
exact rational restatement (tests/exact.py), closed forms and invariants whose
failure would expose a dropped term, a wrong index or a wrong rounding.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


# ----------------------------------------------------------------- encoder

def test_encoder_round_trips_every_finite_code(oracle_mod):
    table = oracle_mod.e4m3_table()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.int64)
    back = oracle_mod.e4m3_encode(table[codes])
    assert np.array_equal(back.astype(np.int64), codes)


def test_encoder_ties_go_to_even_mantissa(oracle_mod):
    table = oracle_mod.e4m3_table()
    pos = [c for c in range(0x7E)]  # 0x00 .. 0x7D and their successors
    mids = np.array([(table[c] + table[c + 1]) / 2 for c in pos])
    got = oracle_mod.e4m3_encode(mids)
    for c, g in zip(pos, got):
        even = c if (c & 1) == 0 else c + 1
        assert g == even, (hex(c), hex(int(g)))
    # and just either side of a midpoint goes to the nearer code
    lo = oracle_mod.e4m3_encode(mids * (1 - 1e-9))
    hi = oracle_mod.e4m3_encode(mids * (1 + 1e-9))
    assert np.array_equal(lo, np.array(pos, np.uint8))
    assert np.array_equal(hi, np.array(pos, np.uint8) + 1)


def test_encoder_saturates_and_maps_nan(oracle_mod):
    got = oracle_mod.e4m3_encode(np.array([448.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf,
                                           np.nan]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def test_encoder_matches_torch_cast_inside_the_range(oracle_mod):
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(20000, generator=g) * 50,
                   torch.randn(20000, generator=g) * 0.01,
                   torch.rand(2000, generator=g) * 896 - 448])
    x = x.clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_mod.e4m3_encode(x.double().numpy())
    assert np.array_equal(got, ref)


# ------------------------------------------------------------ norm + quant

def test_hand_worked_example(oracle_mod):
    with open(os.path.join(GOLDEN, "worked_norm_quant_1x128.json")) as f:
        ex = json.load(f)
    h = ex["hidden"]
    inp = torch.zeros((1, h))
    res = torch.zeros((1, h))
    for j, v in ex["input_nonzero"].items():
        inp[0, int(j)] = v
    for j, v in ex["residual_nonzero"].items():
        res[0, int(j)] = v
    w = torch.full((h,), ex["weight"])
    out = oracle_mod.fused_add_rmsnorm_fp8_block_quant(
        bf16_bits(inp.bfloat16()), bf16_bits(res.bfloat16()), bf16_bits(w.bfloat16()), ex["eps"])
    rsum = bits_to_f64(out["residual_out"][0])
    normed = bits_to_f64(out["normed_out"][0])
    for j in range(h):
        assert rsum[j] == ex["expected_residual_nonzero"].get(str(j), 0.0)
        assert normed[j] == ex["expected_normed_nonzero"].get(str(j), 0.0)
        want = int(ex["expected_codes_nonzero"].get(str(j), "0x00"), 16)
        assert out["out"][0, j] == want, j
    scale = float(out["block_scale"][0, 0])
    assert scale == float(np.float32(9.0625 / 448))
    assert abs(scale - ex["expected_scale_approx"]) < 1e-9


def test_matches_exact_rational_restatement(oracle_mod):
    for seed, rows, hidden, eps, mag in ((11, 3, 256, 1e-6, 1.0), (12, 2, 384, 1e-5, 30.0),
                                         (13, 2, 128, 0.0, 1e-3)):
        inp = bf16_bits(rand_bf16((rows, hidden), seed, mag))
        res = bf16_bits(rand_bf16((rows, hidden), seed + 100, mag))
        w = bf16_bits(rand_bf16((hidden,), seed + 200) .float().abs().add(0.5).bfloat16())
        got = oracle_mod.fused_add_rmsnorm_fp8_block_quant(inp, res, w, eps)
        r_out, n_out, codes, scales = exact.fused_add_rmsnorm_fp8_block_quant(
            inp.tolist(), res.tolist(), w.tolist(), eps)
        assert np.array_equal(got["residual_out"], np.array(r_out, np.uint16))
        assert np.array_equal(got["normed_out"], np.array(n_out, np.uint16))
        assert np.array_equal(got["block_scale"], np.array(scales, np.float32))
        assert np.array_equal(got["out"], np.array(codes, np.uint8))


def test_residual_sum_equals_torch_float32_add_rounded_to_bf16(oracle_mod):
    # The oracle rounds the exact sum once; the FP32 add followed by RNE to BF16
    # (torch's way, and the kernel's) gives the same bits for BF16 operands.
    a = rand_bf16((16, 1024), 21, 10.0)
    b = rand_bf16((16, 1024), 22, 1e-3)  # wide exponent gaps included
    b[::2] = rand_bf16((8, 1024), 23, 1e4)
    got = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bf16_bits(a), bf16_bits(b),
                                                       bf16_bits(torch.ones(1024).bfloat16()))
    want = bf16_bits((a.float() + b.float()).bfloat16())
    assert np.array_equal(got["residual_out"], want)


def test_constant_row_closed_form_with_eps(oracle_mod):
    # x = c everywhere: y = w c / sqrt(c^2 + eps)
    for c, eps in ((0.01, 1e-4), (3.0, 1e-6), (-0.5, 0.25)):
        hidden = 256
        inp = torch.full((1, hidden), c).bfloat16()
        res = torch.zeros((1, hidden)).bfloat16()
        w = torch.full((hidden,), 2.0).bfloat16()
        cv = float(inp[0, 0])
        got = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bf16_bits(inp), bf16_bits(res),
                                                           bf16_bits(w), eps)
        y = 2.0 * cv / math.sqrt(cv * cv + eps)
        want = float(torch.tensor(y, dtype=torch.float64).float().bfloat16())
        assert np.all(bits_to_f64(got["normed_out"]) == want)
        # every element is the block's amax: all codes are +-448
        assert np.all(got["out"] == (0x7E if y > 0 else 0xFE))
        assert np.all(got["block_scale"] == np.float32(abs(want) / 448))


def test_power_of_two_invariances(oracle_mod):
    inp = rand_bf16((4, 512), 31)
    res = rand_bf16((4, 512), 32)
    w = rand_bf16((512,), 33)
    base = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bf16_bits(inp), bf16_bits(res),
                                                        bf16_bits(w), 0.0)
    # scaling the row by 4 leaves the normalised result unchanged (eps = 0)
    up = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bf16_bits(inp * 4), bf16_bits(res * 4),
                                                      bf16_bits(w), 0.0)
    assert np.array_equal(bits_to_f64(up["residual_out"]), 4 * bits_to_f64(base["residual_out"]))
    assert np.array_equal(up["normed_out"], base["normed_out"])
    assert np.array_equal(up["out"], base["out"])
    assert np.array_equal(up["block_scale"], base["block_scale"])
    # doubling the weight doubles normed and the scales; the codes stay
    dw = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bf16_bits(inp), bf16_bits(res),
                                                      bf16_bits(w * 2), 0.0)
    assert np.array_equal(bits_to_f64(dw["normed_out"]), 2 * bits_to_f64(base["normed_out"]))
    assert np.array_equal(dw["block_scale"], 2 * base["block_scale"])
    assert np.array_equal(dw["out"], base["out"])


def test_rows_and_blocks_are_independent(oracle_mod):
    # permuting rows permutes every output; a row's blocks depend on their own
    # 128 columns only through the shared RMS
    inp = rand_bf16((5, 384), 41)
    res = rand_bf16((5, 384), 42)
    w = rand_bf16((384,), 43)
    perm = torch.tensor([3, 0, 4, 1, 2])
    a = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bf16_bits(inp), bf16_bits(res), bf16_bits(w))
    b = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bf16_bits(inp[perm]), bf16_bits(res[perm]),
                                                     bf16_bits(w))
    for key in ("residual_out", "normed_out", "out", "block_scale"):
        assert np.array_equal(b[key], a[key][perm.numpy()]), key


def test_quantisation_bounds_and_zero_blocks(oracle_mod):
    table = oracle_mod.e4m3_table()
    inp = rand_bf16((6, 640), 51, 5.0)
    res = rand_bf16((6, 640), 52, 5.0)
    inp[2, 128:256] = 0
    res[2, 128:256] = 0  # one all-zero block
    w = rand_bf16((640,), 53)
    got = oracle_mod.fused_add_rmsnorm_fp8_block_quant(bf16_bits(inp), bf16_bits(res),
                                                       bf16_bits(w))
    normed = bits_to_f64(got["normed_out"]).reshape(6, 5, 128)
    deq = table[got["out"]].reshape(6, 5, 128) * got["block_scale"][:, :, None].astype(np.float64)
    assert got["block_scale"][2, 1] == 0 and np.all(got["out"][2, 128:256] == 0)
    amax = np.abs(normed).max(axis=2)
    live = amax > 0
    # the largest element of a block maps to +-448 exactly
    codes = got["out"].reshape(6, 5, 128)
    top = np.abs(table[codes]).max(axis=2)
    assert np.all(top[live] == 448.0)
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 for normals, absolute
    # 2^-10 * scale for subnormals, plus the FP32 quotient's rounding
    bound = np.maximum(np.abs(normed) * 2.0 ** -4,
                       2.0 ** -10 * got["block_scale"][:, :, None]) * (1 + 1e-6)
    assert np.all(np.abs(deq - normed) <= bound)
