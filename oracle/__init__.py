"""CPU oracle for the FP8 (E4M3) groupwise-scaled NT GEMM — TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The CUDA library never does: it shares no code with
the oracle, and the product path fails instead of falling back to it.

The arithmetic lives in ``oracle.c`` (plain C, FP64, one rounding); this module
only marshals numpy arrays (or CPU torch tensors) into it.  It follows the MATE
page "FlashInfer Wrapper APIs", section GEMM: ``gemm_fp8_nt_groupwise``,
``group_deepgemm_fp8_nt_groupwise`` and ``batch_deepgemm_fp8_nt_groupwise``;
and section Norm: ``fused_add_rmsnorm_fp8_block_quant`` (the producer of the
GEMM's FP8 activations and their 1 x 128 scales); and the DeepSeek FP8
block-scale MoE layer of the "flashinfer-rs" page built from the grouped GEMM.
"""
import ctypes

import numpy as np

from . import build as _build

OUT_BF16 = 0
OUT_F16 = 1
FP8_E4M3 = 0
FP8_E5M2 = 1
SCALE_K_MAJOR = 0
SCALE_MN_MAJOR = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.oracle_e4m3_table.argtypes = [P]
        lib.oracle_e4m3_table.restype = None
        lib.oracle_round.argtypes = [P, I64, I, P, P]
        lib.oracle_round.restype = None
        lib.oracle_gemm_nt_groupwise.argtypes = [P, P, P, P, I64, I64, I64, I, I, P, P]
        lib.oracle_gemm_nt_groupwise_at.argtypes = [P, P, P, P, I64, I64, I64, I, I,
                                                    P, P, I64, P, P]
        lib.oracle_group_gemm_contiguous.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                                     P, P, P]
        lib.oracle_group_gemm_contiguous_at.argtypes = [P, P, P, P, P, I64, I64, I64,
                                                        I64, P, P, I64, P, P, P]
        lib.oracle_batch_gemm_masked.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                                 P, P, P]
        lib.oracle_batch_gemm_masked_at.argtypes = [P, P, P, P, P, I64, I64, I64, I64,
                                                    P, P, P, I64, P, P, P]
        lib.oracle_e4m3_encode.argtypes = [P, I64, P]
        lib.oracle_e4m3_encode.restype = None
        lib.oracle_fused_add_rmsnorm_fp8_block_quant.argtypes = [
            P, P, P, ctypes.c_double, I64, I64, P, P, P, P]
        lib.oracle_quant_1x128.argtypes = [P, I64, I64, P, P]
        lib.oracle_quant_1x128.restype = None
        lib.oracle_moe_deepseek_fp8_block_scale.argtypes = [P, P, P, P, P, P, I64, I64, I64,
                                                            I64, I64, P]
        lib.oracle_moe_swiglu_quant.argtypes = [P, I64, I64, P, P]
        lib.oracle_moe_combine.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_e5m2_table.argtypes = [P]
        lib.oracle_e5m2_table.restype = None
        lib.oracle_bmm_fp8.argtypes = [P, P, I, I, P, I, P, I, I64, I64, I64, I64, I, P, P]
        for f in ("oracle_gemm_nt_groupwise", "oracle_gemm_nt_groupwise_at",
                  "oracle_bmm_fp8",
                  "oracle_fused_add_rmsnorm_fp8_block_quant",
                  "oracle_moe_deepseek_fp8_block_scale",
                  "oracle_moe_swiglu_quant", "oracle_moe_combine",
                  "oracle_group_gemm_contiguous", "oracle_group_gemm_contiguous_at",
                  "oracle_batch_gemm_masked", "oracle_batch_gemm_masked_at",
                  "oracle_num_threads"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _arr(x, dtype):
    """A C-contiguous numpy array of `dtype` viewing or copying `x`."""
    if hasattr(x, "detach"):  # torch tensor
        t = x.detach().cpu().contiguous()
        if t.element_size() == 1 and dtype == np.uint8:
            import torch
            t = t.view(torch.uint8)
        if t.element_size() == 2 and dtype == np.uint16:  # BF16/FP16 encodings
            import torch
            x = t.view(torch.int16).numpy().view(np.uint16)
        else:
            x = t.numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != dtype:
        if dtype == np.uint8:
            raise TypeError("E4M3 operands must be 1-byte codes, got %s" % a.dtype)
        a = a.astype(dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data


def _check(rc, what):
    if rc == -2:
        raise ValueError("%s: m_indices violates the page's contiguous-layout "
                         "precondition" % what)
    if rc != 0:
        raise ValueError("%s: invalid arguments" % what)


def num_threads():
    return _load().oracle_num_threads()


def e4m3_table():
    """The 256 E4M3 code values (FP64), NaN at 0x7F and 0xFF."""
    out = np.empty(256, np.float64)
    _load().oracle_e4m3_table(out.ctypes.data)
    return out


def round_to(x, out_dtype=OUT_BF16):
    """Round FP64 values once (nearest, ties to even) to BF16/FP16.

    Returns ``(rounded_values_f64, bits_u16)``.
    """
    x = _arr(x, np.float64)
    y = np.empty_like(x)
    bits = np.empty(x.shape, np.uint16)
    _load().oracle_round(x.ctypes.data, x.size, out_dtype, y.ctypes.data,
                         bits.ctypes.data)
    return y, bits


def gemm_nt_groupwise(a, b, a_scale, b_scale, scale_major=SCALE_K_MAJOR,
                      out_dtype=OUT_BF16):
    """Dense form: returns ``(ref_f64 (m,n), bits_u16 (m,n))``."""
    a, b = _arr(a, np.uint8), _arr(b, np.uint8)
    sa, sb = _arr(a_scale, np.float32), _arr(b_scale, np.float32)
    m, k = a.shape
    n = b.shape[0]
    ref = np.empty((m, n), np.float64)
    bits = np.empty((m, n), np.uint16)
    rc = _load().oracle_gemm_nt_groupwise(_p(a), _p(b), _p(sa), _p(sb), m, n, k,
                                          scale_major, out_dtype, _p(ref), _p(bits))
    _check(rc, "gemm_nt_groupwise")
    return ref, bits


def gemm_nt_groupwise_at(a, b, a_scale, b_scale, rows, cols,
                         scale_major=SCALE_K_MAJOR, out_dtype=OUT_BF16):
    """Dense form at positions (rows[s], cols[s]): ``(ref_f64, bits_u16)``."""
    a, b = _arr(a, np.uint8), _arr(b, np.uint8)
    sa, sb = _arr(a_scale, np.float32), _arr(b_scale, np.float32)
    rows, cols = _arr(rows, np.int64).ravel(), _arr(cols, np.int64).ravel()
    m, k = a.shape
    n = b.shape[0]
    ref = np.empty(rows.size, np.float64)
    bits = np.empty(rows.size, np.uint16)
    rc = _load().oracle_gemm_nt_groupwise_at(
        _p(a), _p(b), _p(sa), _p(sb), m, n, k, scale_major, out_dtype,
        _p(rows), _p(cols), rows.size, _p(ref), _p(bits))
    _check(rc, "gemm_nt_groupwise_at")
    return ref, bits


def group_gemm_contiguous(a, b, a_scale, b_scale, m_indices):
    """Contiguous grouped form: ``(ref_f64, bits_u16, written_bool)``, (m,n)."""
    a, b = _arr(a, np.uint8), _arr(b, np.uint8)
    sa, sb = _arr(a_scale, np.float32), _arr(b_scale, np.float32)
    mi = _arr(m_indices, np.int32)
    m, k = a.shape
    g, n = b.shape[0], b.shape[1]
    ref = np.zeros((m, n), np.float64)
    bits = np.zeros((m, n), np.uint16)
    written = np.zeros((m, n), np.uint8)
    rc = _load().oracle_group_gemm_contiguous(
        _p(a), _p(b), _p(sa), _p(sb), _p(mi), m, n, k, g, _p(ref), _p(bits),
        _p(written))
    _check(rc, "group_gemm_contiguous")
    return ref, bits, written.astype(bool)


def group_gemm_contiguous_at(a, b, a_scale, b_scale, m_indices, rows, cols):
    a, b = _arr(a, np.uint8), _arr(b, np.uint8)
    sa, sb = _arr(a_scale, np.float32), _arr(b_scale, np.float32)
    mi = _arr(m_indices, np.int32)
    rows, cols = _arr(rows, np.int64).ravel(), _arr(cols, np.int64).ravel()
    m, k = a.shape
    g, n = b.shape[0], b.shape[1]
    ref = np.zeros(rows.size, np.float64)
    bits = np.zeros(rows.size, np.uint16)
    written = np.zeros(rows.size, np.uint8)
    rc = _load().oracle_group_gemm_contiguous_at(
        _p(a), _p(b), _p(sa), _p(sb), _p(mi), m, n, k, g, _p(rows), _p(cols),
        rows.size, _p(ref), _p(bits), _p(written))
    _check(rc, "group_gemm_contiguous_at")
    return ref, bits, written.astype(bool)


def batch_gemm_masked(a, b, a_scale, b_scale, masked_m):
    """Masked batched form: ``(ref_f64, bits_u16, written_bool)``, (G,max_m,n)."""
    a, b = _arr(a, np.uint8), _arr(b, np.uint8)
    sa, sb = _arr(a_scale, np.float32), _arr(b_scale, np.float32)
    mm = _arr(masked_m, np.int32)
    g, max_m, k = a.shape
    n = b.shape[1]
    ref = np.zeros((g, max_m, n), np.float64)
    bits = np.zeros((g, max_m, n), np.uint16)
    written = np.zeros((g, max_m, n), np.uint8)
    rc = _load().oracle_batch_gemm_masked(
        _p(a), _p(b), _p(sa), _p(sb), _p(mm), g, max_m, n, k, _p(ref), _p(bits),
        _p(written))
    _check(rc, "batch_gemm_masked")
    return ref, bits, written.astype(bool)


def batch_gemm_masked_at(a, b, a_scale, b_scale, masked_m, groups, rows, cols):
    a, b = _arr(a, np.uint8), _arr(b, np.uint8)
    sa, sb = _arr(a_scale, np.float32), _arr(b_scale, np.float32)
    mm = _arr(masked_m, np.int32)
    groups = _arr(groups, np.int64).ravel()
    rows, cols = _arr(rows, np.int64).ravel(), _arr(cols, np.int64).ravel()
    g, max_m, k = a.shape
    n = b.shape[1]
    ref = np.zeros(rows.size, np.float64)
    bits = np.zeros(rows.size, np.uint16)
    written = np.zeros(rows.size, np.uint8)
    rc = _load().oracle_batch_gemm_masked_at(
        _p(a), _p(b), _p(sa), _p(sb), _p(mm), g, max_m, n, k, _p(groups),
        _p(rows), _p(cols), rows.size, _p(ref), _p(bits), _p(written))
    _check(rc, "batch_gemm_masked_at")
    return ref, bits, written.astype(bool)


def e4m3_encode(x):
    """E4M3 codes (uint8) of FP64 values: round to nearest even, saturate to
    +-448, NaN -> 0x7F."""
    x = _arr(x, np.float64)
    codes = np.empty(x.shape, np.uint8)
    _load().oracle_e4m3_encode(x.ctypes.data, x.size, codes.ctypes.data)
    return codes


def fused_add_rmsnorm_fp8_block_quant(input_bits, residual_bits, weight_bits, eps=1e-6):
    """Fused add + RMSNorm + 1 x 128 FP8 quantisation of BF16 rows.

    Arguments are the 16-bit encodings of BF16 tensors: input and residual
    (rows, hidden), weight (hidden).  Returns a dict with ``residual_out`` and
    ``normed_out`` (uint16 encodings, (rows, hidden)), ``out`` (E4M3 codes,
    (rows, hidden)) and ``block_scale`` (float32, (rows, hidden // 128)).
    """
    x = _arr(input_bits, np.uint16)
    r = _arr(residual_bits, np.uint16)
    w = _arr(weight_bits, np.uint16)
    rows, hidden = x.shape
    if r.shape != x.shape or w.shape != (hidden,):
        raise ValueError("shape mismatch")
    res = dict(residual_out=np.empty((rows, hidden), np.uint16),
               normed_out=np.empty((rows, hidden), np.uint16),
               out=np.empty((rows, hidden), np.uint8),
               block_scale=np.empty((rows, hidden // 128 if hidden % 128 == 0 else 0),
                                    np.float32))
    rc = _load().oracle_fused_add_rmsnorm_fp8_block_quant(
        _p(x), _p(r), _p(w), float(eps), rows, hidden, _p(res["residual_out"]),
        _p(res["normed_out"]), _p(res["out"]), _p(res["block_scale"]))
    _check(rc, "fused_add_rmsnorm_fp8_block_quant")
    return res


def quantize_output_e4m3(ref, output_scale):
    """FP8 output of gemm_fp8_nt_groupwise with output_scale (MATE page
    "FlashInfer Wrapper APIs", section GEMM): E4M3 codes of R / s, R the exact
    (FP64) result and s the FP32 output scale, rounded to nearest even and
    saturated to +-448 — the scale multiplies codes back into values, as a_scale
    and b_scale do."""
    r = np.asarray(ref, np.float64)
    return e4m3_encode(r / float(np.float32(output_scale)))


def quant_1x128(x):
    """Row-major 1 x 128 E4M3 quantisation of FP64 values (rows, cols):
    returns (codes uint8 (rows, cols), scales float32 (rows, cols // 128))."""
    x = _arr(x, np.float64)
    rows, cols = x.shape
    if cols % 128:
        raise ValueError("cols must be a multiple of 128")
    codes = np.empty((rows, cols), np.uint8)
    scales = np.empty((rows, cols // 128), np.float32)
    _load().oracle_quant_1x128(x.ctypes.data, rows, cols, codes.ctypes.data, scales.ctypes.data)
    return codes, scales


def moe_deepseek_fp8_block_scale(input_bits, token_selected, w1, w2, s1, s2):
    """DeepSeek FP8 block-scale MoE layer (see oracle.h): BF16 input
    encodings (tokens, hidden), int32 token_selected (tokens, top_k), E4M3
    fc1 (E, 2*inter, hidden) and fc2 (E, hidden, inter) with their FP32 block
    scales.  Returns the BF16 encodings of out (tokens, hidden)."""
    x = _arr(input_bits, np.uint16)
    ts = _arr(token_selected, np.int32)
    w1, w2 = _arr(w1, np.uint8), _arr(w2, np.uint8)
    s1, s2 = _arr(s1, np.float32), _arr(s2, np.float32)
    tokens, hidden = x.shape
    top_k = ts.shape[1]
    e, two_i, h2 = w1.shape
    inter = two_i // 2
    if h2 != hidden or w2.shape != (e, hidden, inter) or ts.shape[0] != tokens:
        raise ValueError("shape mismatch")
    if s1.shape != (e, two_i // 128, hidden // 128) or s2.shape != (e, hidden // 128, inter // 128):
        raise ValueError("scale shape mismatch")
    out = np.empty((tokens, hidden), np.uint16)
    rc = _load().oracle_moe_deepseek_fp8_block_scale(
        _p(x), _p(ts), _p(w1), _p(w2), _p(s1), _p(s2), tokens, e, top_k, hidden, inter, _p(out))
    if rc == -2:
        raise ValueError("moe: token_selected holds an expert id outside [-1, num_experts)")
    _check(rc, "moe_deepseek_fp8_block_scale")
    return out


def moe_swiglu_quant(h_bits):
    """The MoE layer's SwiGLU step on given fc1 outputs: h (rows, 2*inter) BF16
    encodings (gate, then up).  act = silu(gate) * up in FP64, then its 1 x 128
    quantisation; returns (codes uint8 (rows, inter), scales float32 (rows,
    inter // 128))."""
    h = _arr(h_bits, np.uint16)
    rows, two_i = h.shape
    inter = two_i // 2
    codes = np.empty((rows, inter), np.uint8)
    scales = np.empty((rows, inter // 128 if inter % 128 == 0 else 0), np.float32)
    rc = _load().oracle_moe_swiglu_quant(_p(h), rows, inter, _p(codes), _p(scales))
    _check(rc, "moe_swiglu_quant")
    return codes, scales


def moe_combine(y_bits, row_of):
    """The MoE layer's combine step on given fc2 outputs: y (rows, hidden) BF16
    encodings, row_of (tokens, top_k) int32 rows of y (-1: empty slot).
    Returns the BF16 encodings of out (tokens, hidden): each token's rows summed
    exactly and rounded once."""
    y = _arr(y_bits, np.uint16)
    ro = _arr(row_of, np.int32)
    tokens, top_k = ro.shape
    hidden = y.shape[1]
    if ro.size and (ro.max() >= y.shape[0]):
        raise ValueError("row_of points past the rows of y")
    out = np.empty((tokens, hidden), np.uint16)
    rc = _load().oracle_moe_combine(_p(y), _p(ro), tokens, top_k, hidden, _p(out))
    _check(rc, "moe_combine")
    return out


def e5m2_table():
    """The 256 E5M2 code values (FP64): +-inf at 0x7C/0xFC, NaN at 0x7D-0x7F, 0xFD-0xFF."""
    out = np.empty(256, np.float64)
    _load().oracle_e5m2_table(out.ctypes.data)
    return out


def bmm_fp8(a, b, a_scale, b_scale, a_fmt=FP8_E4M3, b_fmt=FP8_E4M3, out_dtype=OUT_BF16):
    """bmm_fp8 (section GEMM): A (batch, m, k), B (batch, k, n) FP8 codes; each
    scale a one-element (tensorwise) or channelwise array — a_scale (batch, m, 1),
    b_scale (batch, 1, n).  Returns (ref_f64, bits_u16), both (batch, m, n)."""
    a, b = _arr(a, np.uint8), _arr(b, np.uint8)
    sa, sb = _arr(a_scale, np.float32), _arr(b_scale, np.float32)
    batch, m, k = a.shape
    n = b.shape[2]
    if b.shape[:2] != (batch, k):
        raise ValueError("B must be (batch, k, n)")
    a_ch = sa.size != 1
    b_ch = sb.size != 1
    if a_ch and sa.shape != (batch, m, 1):
        raise ValueError("channelwise a_scale must be (batch, m, 1)")
    if b_ch and sb.shape != (batch, 1, n):
        raise ValueError("channelwise b_scale must be (batch, 1, n)")
    ref = np.empty((batch, m, n), np.float64)
    bits = np.empty((batch, m, n), np.uint16)
    rc = _load().oracle_bmm_fp8(_p(a), _p(b), int(a_fmt), int(b_fmt), _p(sa), int(a_ch), _p(sb),
                                int(b_ch), batch, m, n, k, int(out_dtype), _p(ref), _p(bits))
    _check(rc, "bmm_fp8")
    return ref, bits
