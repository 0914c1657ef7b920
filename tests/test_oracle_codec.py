"""Pins of the oracle's E4M3 decode and its final rounding (CPU only).

The decode table is checked against hand-worked codes, against the exact
restatement in ``tests/exact.py`` and against torch's own float8_e4m3fn
conversion; the rounding against numpy's float64->float16 cast, torch's
float32->bfloat16 cast and an exact rational rounding.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_decode_table_matches_hand_worked_codes(oracle_mod):
    table = oracle_mod.e4m3_table()
    seen = 0
    with open(os.path.join(GOLDEN, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code_s, val_s = line.split()
            code = int(code_s, 16)
            if val_s == "nan":
                assert math.isnan(table[code])
            else:
                v = float(val_s)
                assert table[code] == v
                assert math.copysign(1.0, table[code]) == math.copysign(1.0, v)
            seen += 1
    assert seen >= 20


def test_decode_table_matches_exact_fields(oracle_mod):
    table = oracle_mod.e4m3_table()
    for c in range(256):
        v = exact.e4m3_value(c)
        if v is None:
            assert math.isnan(table[c]), hex(c)
        else:
            assert Fraction(float(table[c])) == v, hex(c)
    assert int(np.isnan(table).sum()) == 2  # 0x7F and 0xFF only: no infinities


def test_decode_table_matches_torch_float8(oracle_mod):
    table = oracle_mod.e4m3_table()
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ref) & np.isnan(table)
    assert np.array_equal(ref[~both_nan], table[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(table))


def test_decode_range_properties(oracle_mod):
    t = oracle_mod.e4m3_table()
    finite = t[~np.isnan(t)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    pos = finite[finite > 0]
    assert pos.min() == 2.0 ** -9
    # every value is an integer number of 2^-9 units (block sums are exact)
    units = finite * 512.0
    assert np.array_equal(units, np.round(units))


def _edge_doubles():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, -65520.0, 70000.0,
            2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26,
            3 * 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
            1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40,
            3.3895313892515355e38, 3.3961775292304776e38, 3.4e38, 1e39, 1e-39,
            2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134, 2.0 ** -126, float("inf"),
            float("-inf")]
    return np.array(vals, dtype=np.float64)


def test_round_f16_matches_numpy(oracle_mod):
    rng = np.random.default_rng(1)
    x = np.concatenate([
        _edge_doubles(),
        rng.standard_normal(20000) * np.exp2(rng.uniform(-30, 18, 20000)),
        # exact ties between two FP16 neighbours
        (np.arange(-3000, 3000) + 0.5) * 2.0 ** -10,
        (np.arange(0, 2000) + 0.5) * 2.0 ** -24,
    ])
    _, bits = oracle_mod.round_to(x, oracle_mod.OUT_F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(bits, ref)


def test_round_bf16_matches_torch_on_float32_inputs(oracle_mod):
    # For values that are FP32-representable, FP32->BF16 is a single rounding.
    g = torch.Generator().manual_seed(2)
    x32 = torch.randn(50000, generator=g) * torch.exp2(torch.empty(50000).uniform_(-130, 120, generator=g))
    ties = (torch.arange(-4000, 4000, dtype=torch.float32) * 2 + 1) * 2.0 ** -8  # odd/256: tie
    x32 = torch.cat([x32, ties, torch.tensor(_edge_doubles(), dtype=torch.float32)])
    ref = x32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    _, bits = oracle_mod.round_to(x32.double().numpy(), oracle_mod.OUT_BF16)
    assert np.array_equal(bits, ref)


@pytest.mark.parametrize("fmt,code", [("bf16", 0), ("f16", 1)])
def test_round_matches_exact_rational_rounding(oracle_mod, fmt, code):
    rng = np.random.default_rng(3)
    x = np.concatenate([_edge_doubles()[:-2],
                        rng.standard_normal(3000) * np.exp2(rng.uniform(-140, 125, 3000))])
    y, _ = oracle_mod.round_to(x, code)
    for xi, yi in zip(x, y):
        want = exact.round_exact(Fraction(float(xi)), fmt)
        if isinstance(want, float):
            assert yi == want, (xi, yi, want)
        else:
            assert Fraction(float(yi)) == want, (xi, yi, want)
