"""Exact rational restatements of the groupwise FP8 GEMM and of the fused
add-RMSNorm + 1 x 128 FP8 quantisation, for tiny shapes.

An independent second implementation used to pin the C oracle: E4M3 decoded
from its bit fields into ``fractions.Fraction``, block sums in Python integers
(every E4M3 value is an integer multiple of 2^-9), scales converted exactly
from FP32, and the final value rounded to BF16/FP16 by exact comparison.  It
follows the MATE page "FlashInfer Wrapper APIs", section GEMM
(gemm_fp8_nt_groupwise and its grouped and masked forms).
"""
from fractions import Fraction

import numpy as np

FORMATS = {
    # significand bits (with the implicit one), smallest normal exponent,
    # largest finite value
    "bf16": (8, -126, Fraction(2 ** 8 - 1, 2 ** 7) * Fraction(2) ** 127),
    "f16": (11, -14, Fraction(65504)),
    "f32": (24, -126, Fraction(2 ** 24 - 1, 2 ** 23) * Fraction(2) ** 127),
    "e4m3": (4, -6, Fraction(448)),
}


def e4m3_value(code):
    """Exact value of an E4M3 (float8_e4m3fn) code, None for NaN."""
    s, e, f = (code >> 7) & 1, (code >> 3) & 0xF, code & 7
    if e == 0xF and f == 7:
        return None
    if e == 0:
        v = Fraction(f, 8) * Fraction(1, 2 ** 6)
    else:
        v = (1 + Fraction(f, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def e4m3_units(code):
    """The code's value in units of 2^-9 (an integer)."""
    v = e4m3_value(code) * 512
    assert v.denominator == 1
    return int(v)


UNITS = np.array([e4m3_units(c) if e4m3_value(c) is not None else 0
                  for c in range(256)], dtype=np.int64)


def floor_log2(x):
    """floor(log2(x)) of a positive Fraction, exactly."""
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    return e


def round_exact(x, fmt):
    """Nearest value of format `fmt` to the Fraction x, ties to even.

    Returns a Fraction, or +-inf (float) on overflow.
    """
    p, emin, maxf = FORMATS[fmt]
    if x == 0:
        return Fraction(0)
    lead = max(floor_log2(abs(x)), emin)
    quantum = Fraction(2) ** (lead - p + 1)
    y = round(x / quantum) * quantum  # Fraction.__round__ ties to even
    if abs(y) > maxf:
        return float("inf") if x > 0 else float("-inf")
    return y


def block_sums(a_codes, b_codes):
    """Integer block sums P*2^18, shape (rows_a, rows_b, k/128)."""
    a = UNITS[np.asarray(a_codes, dtype=np.int64)]
    b = UNITS[np.asarray(b_codes, dtype=np.int64)]
    kb = a.shape[1] // 128
    out = np.empty((a.shape[0], b.shape[0], kb), dtype=object)
    for t in range(kb):
        blk = a[:, t * 128:(t + 1) * 128] @ b[:, t * 128:(t + 1) * 128].T
        out[:, :, t] = blk.astype(object)
    return out


def dense(a_codes, b_codes, sa, sb, with_abs=False):
    """Exact R(i,j) for K-major scales sa (m,KB), sb (n/128,KB) (FP32 arrays).

    With `with_abs`, also the sums of |P * sa * sb| over K blocks (the scale of
    the rounding error an FP64 evaluation may make)."""
    P = block_sums(a_codes, b_codes)
    m, n, kb = P.shape
    unit = Fraction(1, 2 ** 18)
    sa = [[Fraction(float(v)) for v in row] for row in np.asarray(sa, np.float32)]
    sb = [[Fraction(float(v)) for v in row] for row in np.asarray(sb, np.float32)]
    R = [[None] * n for _ in range(m)]
    A = [[None] * n for _ in range(m)]
    for i in range(m):
        for j in range(n):
            jb = j // 128
            terms = [int(P[i, j, t]) * unit * sa[i][t] * sb[jb][t] for t in range(kb)]
            R[i][j] = sum(terms, Fraction(0))
            A[i][j] = sum((abs(x) for x in terms), Fraction(0))
    return (R, A) if with_abs else R


def bf16_value(bits):
    """Exact value of a BF16 encoding (finite values only)."""
    bits = int(bits)
    s, e, f = bits >> 15, (bits >> 7) & 0xFF, bits & 0x7F
    assert e != 0xFF
    v = Fraction(f, 128) * Fraction(2) ** -126 if e == 0 else \
        (1 + Fraction(f, 128)) * Fraction(2) ** (e - 127)
    return -v if s else v


def e4m3_code(v):
    """E4M3 code of a value on the E4M3 grid with |v| <= 448."""
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        if e4m3_value(c) == v and (v != 0 or c == 0):
            return c
    raise ValueError(v)


def fused_add_rmsnorm_fp8_block_quant(input_bits, residual_bits, weight_bits, eps):
    """fused_add_rmsnorm_fp8_block_quant (MATE page "FlashInfer Wrapper APIs",
    section Norm) in exact arithmetic: the add and the sum of squares exactly,
    the reciprocal square root to 80 significant digits (a BF16 rounding decision
    is wrong only if the value lies within 1e-70 of a tie), every rounding by
    exact comparison.  Returns (residual_bits, normed_bits, codes, scales) as
    nested lists."""
    from decimal import Decimal, getcontext
    getcontext().prec = 80
    rows, hidden = len(input_bits), len(input_bits[0])
    w = [bf16_value(b) for b in weight_bits]
    res_out, normed_out, codes, scales = [], [], [], []
    for i in range(rows):
        x = [round_exact(bf16_value(a) + bf16_value(b), "bf16")
             for a, b in zip(input_bits[i], residual_bits[i])]
        ms = sum(v * v for v in x) / hidden + Fraction(eps)
        r = 1 / Decimal(ms.numerator).__truediv__(Decimal(ms.denominator)).sqrt()
        y = [round_exact(Fraction(Decimal(v.numerator) / Decimal(v.denominator) * r
                                  * Decimal(wj.numerator) / Decimal(wj.denominator)), "bf16")
             for v, wj in zip(x, w)]
        res_out.append([bf16_bits(v) for v in x])
        normed_out.append([bf16_bits(v) for v in y])
        crow, srow = [], []
        for b0 in range(0, hidden, 128):
            blk = y[b0:b0 + 128]
            amax = max(abs(v) for v in blk)
            scale = round_exact(amax / 448, "f32")
            srow.append(float(scale))
            for v in blk:
                if amax == 0:
                    crow.append(0)
                    continue
                q = round_exact(v / scale, "f32")
                e = round_exact(q, "e4m3")
                if isinstance(e, float) or abs(e) > 448:  # saturate
                    e = Fraction(448) if q > 0 else Fraction(-448)
                c = e4m3_code(e) if e != 0 else (0x80 if v < 0 else 0)
                crow.append(c)
        codes.append(crow)
        scales.append(srow)
    return res_out, normed_out, codes, scales


def bf16_bits(v):
    """BF16 encoding of a value on the BF16 grid."""
    import struct
    f = struct.pack(">f", float(v))
    return int.from_bytes(f[:2], "big")


def e5m2_value(code):
    """Exact value of an E5M2 (float8_e5m2) code, None for NaN or infinity."""
    s, e, f = (code >> 7) & 1, (code >> 2) & 0x1F, code & 3
    if e == 0x1F:
        return None
    if e == 0:
        v = Fraction(f, 4) * Fraction(1, 2 ** 14)
    else:
        v = (1 + Fraction(f, 4)) * Fraction(2) ** (e - 15)
    return -v if s else v


def bmm(a_codes, b_codes, a_fmt, b_fmt, sa, sb, fmt):
    """bmm_fp8 (MATE page "FlashInfer Wrapper APIs", section GEMM) exactly:
    out[bb][i][j] = round((sum_t A[bb][i][t] * B[bb][t][j]) * sa * sb) with sa,
    sb the FP32 scales of row i / column j (or one tensorwise value each)."""
    dec = {0: e4m3_value, 1: e5m2_value}
    batch, m, k = a_codes.shape
    n = b_codes.shape[2]
    out = np.empty((batch, m, n), dtype=object)
    for bb in range(batch):
        for i in range(m):
            for j in range(n):
                acc = sum(dec[a_fmt](int(a_codes[bb, i, t])) * dec[b_fmt](int(b_codes[bb, t, j]))
                          for t in range(k))
                s_a = Fraction(float(sa.flat[0] if sa.size == 1 else sa[bb, i, 0]))
                s_b = Fraction(float(sb.flat[0] if sb.size == 1 else sb[bb, 0, j]))
                out[bb, i, j] = round_exact(acc * s_a * s_b, fmt)
    return out
