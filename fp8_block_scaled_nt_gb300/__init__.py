"""FP8 (E4M3) groupwise-scaled NT GEMM for GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/fp8g.h``.  It only marshals
arguments — tensor pointers, sizes, the current CUDA stream — and raises on a
non-zero status; every step of the computation runs in the library's CUDA
kernels.  If ``libfp8g.so`` is missing, calls fail: there is no other path.

Two layers of GEMM calls, both following the MATE page "FlashInfer Wrapper
APIs", section GEMM:

* ``fp8_gemm_nt_groupwise``, ``fp8_group_gemm_contiguous``,
  ``fp8_batch_gemm_masked`` — the C entry points, same names, taking tensors
  and a preallocated ``out``;
* ``gemm_fp8_nt_groupwise``, ``group_deepgemm_fp8_nt_groupwise``,
  ``batch_deepgemm_fp8_nt_groupwise`` — the page's own signatures, which
  allocate ``out`` when it is omitted and return it.

and ``fused_add_rmsnorm_fp8_block_quant`` (section Norm, same name and argument
order as the page), which produces the GEMMs' FP8 activations and K-major
1 x 128 scales.

E4M3 operands may be ``torch.float8_e4m3fn`` or ``torch.uint8`` (raw codes).
"""
import ctypes
import os

__all__ = [
    "Fp8gError", "load", "last_error", "get_device_status", "get_stream_status",
    "moe_workspace_layout",
    "fp8_gemm_nt_groupwise", "fp8_group_gemm_contiguous", "fp8_batch_gemm_masked",
    "gemm_fp8_nt_groupwise", "group_deepgemm_fp8_nt_groupwise",
    "batch_deepgemm_fp8_nt_groupwise", "fused_add_rmsnorm_fp8_block_quant",
    "fused_moe_deepseek_fp8_block_scale", "moe_workspace_size",
    "fused_moe_deepseek_fp8_block_scale_noalloc", "MOE_STATIC_SCRATCH_BYTES", "bmm_fp8",
    "OK", "ERR_INVALID_ARGUMENT", "ERR_UNSUPPORTED", "ERR_ARCH", "ERR_CUDA", "ERR_TIMEOUT",
    "DEVICE_TIMEOUT", "DEVICE_BAD_M_INDICES", "DEVICE_MASKED_M_CLAMPED",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp8g.so")

OK, ERR_INVALID_ARGUMENT, ERR_UNSUPPORTED, ERR_ARCH, ERR_CUDA, ERR_TIMEOUT = range(6)
STATUS_NAMES = {0: "FP8G_OK", 1: "FP8G_ERR_INVALID_ARGUMENT", 2: "FP8G_ERR_UNSUPPORTED",
                3: "FP8G_ERR_ARCH", 4: "FP8G_ERR_CUDA", 5: "FP8G_ERR_TIMEOUT"}
SCALE_K_MAJOR, SCALE_MN_MAJOR = 0, 1
OUT_BF16, OUT_F16, OUT_E4M3 = 0, 1, 2
DEVICE_TIMEOUT, DEVICE_BAD_M_INDICES, DEVICE_MASKED_M_CLAMPED = 0x1, 0x2, 0x4
MOE_STATIC_SCRATCH_BYTES = 64 << 20  # FP8G_MOE_STATIC_SCRATCH_BYTES


class Fp8gError(RuntimeError):
    def __init__(self, status, func, message):
        super().__init__("%s: %s: %s" % (func, STATUS_NAMES.get(status, status), message))
        self.status = status


_lib = None


def load():
    """Load ``libfp8g.so`` (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("fp8g CUDA library not built (%s missing); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.fp8_gemm_nt_groupwise.argtypes = [P, P, P, P, P, I, P, I64, I64, I64, I, I, I, I, I, P]
    lib.fp8_group_gemm_contiguous.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, P]
    lib.fp8_batch_gemm_masked.argtypes = [P, P, P, P, P, I64, P, I64, I64, I64, I64, P]
    lib.fp8g_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), I]
    lib.bmm_fp8.argtypes = [P, P, I, I, P, I, P, I, P, I, I64, I64, I64, I64, P]
    lib.fused_add_rmsnorm_fp8_block_quant.argtypes = [P, P, P, P, P, P, ctypes.c_float, I64,
                                                      I64, P]
    lib.fused_moe_deepseek_fp8_block_scale_workspace_size.argtypes = [I64, I64, I64, I64, I64]
    lib.fused_moe_deepseek_fp8_block_scale_workspace_size.restype = ctypes.c_size_t
    lib.fused_moe_deepseek_fp8_block_scale.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, I64,
                                                       I64, P, ctypes.c_size_t, P]
    lib.fused_moe_deepseek_fp8_block_scale_noalloc.argtypes = [P, P, P, P, P, P, P, I64, I64,
                                                               I64, I64, I64, P]
    lib.fp8g_get_stream_status.argtypes = [ctypes.POINTER(ctypes.c_uint), I, P]
    lib.fused_moe_deepseek_fp8_block_scale_workspace_layout.argtypes = [
        I64, I64, I64, I64, I64, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_size_t)]
    lib.fp8g_testing_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.fp8g_testing_set_wait_limit_ns.restype = None
    lib.fp8g_testing_last_gemm_cta_pair.argtypes = []
    lib.fp8g_testing_last_gemm_cta_pair.restype = ctypes.c_int
    for f in ("fp8_gemm_nt_groupwise", "fp8_group_gemm_contiguous", "fp8_batch_gemm_masked",
              "fused_add_rmsnorm_fp8_block_quant", "fused_moe_deepseek_fp8_block_scale", "bmm_fp8",
              "fused_moe_deepseek_fp8_block_scale_noalloc", "fp8g_get_device_status",
              "fp8g_get_stream_status", "fused_moe_deepseek_fp8_block_scale_workspace_layout"):
        getattr(lib, f).restype = ctypes.c_int
    lib.fp8g_last_error.argtypes = []
    lib.fp8g_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def last_error():
    return load().fp8g_last_error().decode()


def _raise_on(rc, func):
    if rc != OK:
        raise Fp8gError(rc, func, last_error())


def get_device_status(clear=True):
    """OR of DEVICE_* bits raised by kernels on the current device (synchronises)."""
    v = ctypes.c_uint(0)
    rc = load().fp8g_get_device_status(ctypes.byref(v), 1 if clear else 0)
    if rc not in (OK, ERR_TIMEOUT):
        _raise_on(rc, "fp8g_get_device_status")
    return v.value


def get_stream_status(clear=True, stream=None):
    """The same bits, read in the order of ``stream`` (the current stream when
    omitted): waits for that stream only."""
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    v = ctypes.c_uint(0)
    rc = load().fp8g_get_stream_status(ctypes.byref(v), 1 if clear else 0, stream.cuda_stream)
    if rc not in (OK, ERR_TIMEOUT):
        _raise_on(rc, "fp8g_get_stream_status")
    return v.value


MOE_WORKSPACE_REGIONS = ("m_indices", "row_of", "a1", "a1_scale", "h", "a2", "a2_scale", "y")


def moe_workspace_layout(num_tokens, num_experts, top_k, hidden_size, inter_size):
    """Rows M of the MoE layer's routed layout and the byte offset of each
    workspace region (``MOE_WORKSPACE_REGIONS``; see include/fp8g.h)."""
    rows = ctypes.c_int64(0)
    offs = (ctypes.c_size_t * 8)()
    rc = load().fused_moe_deepseek_fp8_block_scale_workspace_layout(
        num_tokens, num_experts, top_k, hidden_size, inter_size, ctypes.byref(rows), offs)
    _raise_on(rc, "fused_moe_deepseek_fp8_block_scale_workspace_layout")
    return rows.value, dict(zip(MOE_WORKSPACE_REGIONS, (int(o) for o in offs)))


# ------------------------------------------------------------- marshalling

def _torch():
    import torch
    return torch


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _stream_handle(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _e4m3(t, name):
    torch = _torch()
    if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError("%s must be float8_e4m3fn (or uint8 codes), got %s" % (name, t.dtype))
    return t


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _cuda_contig(ts, names):
    dev = None
    for t, nm in zip(ts, names):
        if t is None:
            continue
        _need(t.is_cuda, "%s must be a CUDA tensor" % nm)
        _need(t.is_contiguous(), "%s must be contiguous" % nm)
        if dev is None:
            dev = t.device
        _need(t.device == dev, "%s is on %s, expected %s" % (nm, t.device, dev))
    return dev


def _out_code(dtype):
    torch = _torch()
    if dtype == torch.bfloat16:
        return OUT_BF16
    if dtype == torch.float16:
        return OUT_F16
    if dtype in (torch.float8_e4m3fn, torch.uint8):
        return OUT_E4M3
    raise TypeError("output dtype must be bfloat16, float16 or float8_e4m3fn, got %s" % dtype)


def _check_granularity(g):
    if tuple(g) != (1, 128, 128):
        raise Fp8gError(ERR_UNSUPPORTED, "scale_granularity_mnk",
                        "only (1, 128, 128) is provided, got %s" % (tuple(g),))


# ------------------------------------------------------------- C entry points

def fp8_gemm_nt_groupwise(a, b, a_scale, b_scale, out, scale_major="K", mma_sm=0,
                          scale_granularity_mnk=(1, 128, 128), stream=None, output_scale=None):
    """out (m,n) = a (m,k) @ b (n,k).T with groupwise scales; returns out.

    ``mma_sm``: 0 picks the tile shape (one SM per 128 x 256 tile, or a CTA pair
    per 256 x 256 tile) from the problem size; 1 and 2 force one or the other.
    Results are bit-identical either way.

    ``out`` is BF16/FP16, or E4M3 (``float8_e4m3fn`` or ``uint8`` codes) together
    with ``output_scale``, a one-element float32 device tensor s: out = E4M3(R / s).
    """
    torch = _torch()
    code = _out_code(out.dtype)
    _need((code == OUT_E4M3) == (output_scale is not None),
          "output_scale goes with (and only with) an E4M3 out")
    if output_scale is not None:
        _need(output_scale.dtype == torch.float32 and output_scale.numel() == 1,
              "output_scale must be a one-element float32 tensor")
    _e4m3(a, "a"), _e4m3(b, "b")
    _need(a.dim() == 2 and b.dim() == 2 and out.dim() == 2, "a, b, out must be 2-D")
    m, k = a.shape
    n = b.shape[0]
    _need(b.shape[1] == k, "b must be (n, %d), got %s" % (k, tuple(b.shape)))
    _need(tuple(out.shape) == (m, n), "out must be (%d, %d), got %s" % (m, n, tuple(out.shape)))
    _need(a_scale.dtype == torch.float32 and b_scale.dtype == torch.float32, "scales must be float32")
    kb, nb = k // 128, n // 128
    if b_scale.numel() == 1 and nb * kb != 1:
        # a scalar b_scale (the page allows one: only a non-scalar tensor must be
        # contiguous) scales every block of b alike: it is handed to the library
        # as that value on the whole (n/128, k/128) block grid
        grid = (nb, kb) if scale_major in (None, "K") else (kb, nb)
        b_scale = b_scale.reshape(1, 1).expand(*grid).contiguous()
    if scale_major in (None, "K"):
        sm = SCALE_K_MAJOR
        _need(tuple(a_scale.shape) == (m, kb), "K-major a_scale must be (%d, %d)" % (m, kb))
        _need(tuple(b_scale.shape) == (nb, kb), "K-major b_scale must be (%d, %d)" % (nb, kb))
    elif scale_major == "MN":
        sm = SCALE_MN_MAJOR
        _need(tuple(a_scale.shape) == (kb, m), "MN-major a_scale must be (%d, %d)" % (kb, m))
        _need(tuple(b_scale.shape) == (kb, nb), "MN-major b_scale must be (%d, %d)" % (kb, nb))
    else:
        raise ValueError("scale_major must be 'K', 'MN' or None")
    dev = _cuda_contig((a, b, a_scale, b_scale, out, output_scale),
                       ("a", "b", "a_scale", "b_scale", "out", "output_scale"))
    g = tuple(scale_granularity_mnk)
    rc = load().fp8_gemm_nt_groupwise(
        _ptr(a), _ptr(b), _ptr(a_scale), _ptr(b_scale), _ptr(out), code, _ptr(output_scale),
        m, n, k, sm, g[0], g[1], g[2], int(mma_sm), _stream_handle(stream, dev))
    _raise_on(rc, "fp8_gemm_nt_groupwise")
    return out


def fp8_group_gemm_contiguous(a, b, a_scale, b_scale, m_indices, out, stream=None):
    """out[i] = a[i] @ b[m_indices[i]].T for rows with m_indices != -1."""
    torch = _torch()
    _e4m3(a, "a"), _e4m3(b, "b")
    _need(a.dim() == 2 and b.dim() == 3, "a must be (m, k) and b (num_groups, n, k)")
    m, k = a.shape
    g, n = b.shape[0], b.shape[1]
    _need(b.shape[2] == k, "b must be (G, n, %d)" % k)
    _need(tuple(out.shape) == (m, n) and out.dtype == torch.bfloat16, "out must be bf16 (m, n)")
    _need(tuple(a_scale.shape) == (m, k // 128), "a_scale must be (m, k // 128)")
    _need(tuple(b_scale.shape) == (g, n // 128, k // 128), "b_scale must be (G, n // 128, k // 128)")
    _need(a_scale.dtype == torch.float32 and b_scale.dtype == torch.float32, "scales must be float32")
    _need(m_indices.dtype == torch.int32 and tuple(m_indices.shape) == (m,),
          "m_indices must be int32 (m,)")
    dev = _cuda_contig((a, b, a_scale, b_scale, m_indices, out),
                       ("a", "b", "a_scale", "b_scale", "m_indices", "out"))
    rc = load().fp8_group_gemm_contiguous(
        _ptr(a), _ptr(b), _ptr(a_scale), _ptr(b_scale), _ptr(m_indices), _ptr(out),
        m, n, k, g, _stream_handle(stream, dev))
    _raise_on(rc, "fp8_group_gemm_contiguous")
    return out


def fp8_batch_gemm_masked(a, b, a_scale, b_scale, masked_m, expected_m, out, stream=None):
    """out[g, :masked_m[g]] = a[g, :masked_m[g]] @ b[g].T."""
    torch = _torch()
    _e4m3(a, "a"), _e4m3(b, "b")
    _need(a.dim() == 3 and b.dim() == 3, "a must be (G, max_m, k) and b (G, n, k)")
    g, max_m, k = a.shape
    n = b.shape[1]
    _need(b.shape[0] == g and b.shape[2] == k, "b must be (%d, n, %d)" % (g, k))
    _need(tuple(out.shape) == (g, max_m, n) and out.dtype == torch.bfloat16,
          "out must be bf16 (G, max_m, n)")
    _need(tuple(a_scale.shape) == (g, max_m, k // 128), "a_scale must be (G, max_m, k // 128)")
    _need(tuple(b_scale.shape) == (g, n // 128, k // 128), "b_scale must be (G, n // 128, k // 128)")
    _need(a_scale.dtype == torch.float32 and b_scale.dtype == torch.float32, "scales must be float32")
    _need(masked_m.dtype == torch.int32 and tuple(masked_m.shape) == (g,),
          "masked_m must be int32 (G,)")
    dev = _cuda_contig((a, b, a_scale, b_scale, masked_m, out),
                       ("a", "b", "a_scale", "b_scale", "masked_m", "out"))
    rc = load().fp8_batch_gemm_masked(
        _ptr(a), _ptr(b), _ptr(a_scale), _ptr(b_scale), _ptr(masked_m), int(expected_m),
        _ptr(out), g, max_m, n, k, _stream_handle(stream, dev))
    _raise_on(rc, "fp8_batch_gemm_masked")
    return out


def fused_add_rmsnorm_fp8_block_quant(out, block_scale, normed_out, input, residual, weight,
                                      eps=1e-6, enable_pdl=None, stream=None):
    """residual += input; normed_out = RMSNorm(residual) * weight; out, block_scale =
    row-major 1 x 128 E4M3 quantisation of normed_out (scales are multipliers).

    ``enable_pdl`` is accepted for the page's signature: every launch of this
    library already lets its prologue overlap the previous kernel.
    """
    torch = _torch()
    del enable_pdl
    _e4m3(out, "out")
    _need(input.dim() == 2, "input must be (rows, hidden)")
    rows, hidden = input.shape
    for t, nm in ((input, "input"), (residual, "residual"), (normed_out, "normed_out")):
        _need(t.dtype == torch.bfloat16 and tuple(t.shape) == (rows, hidden),
              "%s must be bfloat16 (%d, %d)" % (nm, rows, hidden))
    _need(weight.dtype == torch.bfloat16 and tuple(weight.shape) == (hidden,),
          "weight must be bfloat16 (%d,)" % hidden)
    _need(tuple(out.shape) == (rows, hidden), "out must be (%d, %d)" % (rows, hidden))
    _need(block_scale.dtype == torch.float32 and tuple(block_scale.shape) == (rows, hidden // 128),
          "block_scale must be float32 (rows, hidden // 128)")
    dev = _cuda_contig((out, block_scale, normed_out, input, residual, weight),
                       ("out", "block_scale", "normed_out", "input", "residual", "weight"))
    rc = load().fused_add_rmsnorm_fp8_block_quant(
        _ptr(out), _ptr(block_scale), _ptr(normed_out), _ptr(input), _ptr(residual),
        _ptr(weight), float(eps), rows, hidden, _stream_handle(stream, dev))
    _raise_on(rc, "fused_add_rmsnorm_fp8_block_quant")


def moe_workspace_size(num_tokens, num_experts, top_k, hidden_size, inter_size):
    """Bytes of device workspace fused_moe_deepseek_fp8_block_scale needs."""
    return int(load().fused_moe_deepseek_fp8_block_scale_workspace_size(
        num_tokens, num_experts, top_k, hidden_size, inter_size))


def _moe_args(input, token_selected, fc1_weights, fc2_weights, out, fc1_scales, fc2_scales):
    """Checks the MoE layer's tensors against one another (the C ABI gets only
    pointers and sizes, so a mismatch must be caught here) and returns
    (T, E, top_k, H, I, device)."""
    torch = _torch()
    _need(input.dim() == 2 and input.dtype == torch.bfloat16, "input must be bfloat16 (T, H)")
    t, hdim = input.shape
    _need(token_selected.dim() == 2 and token_selected.dtype == torch.int32 and
          token_selected.shape[0] == t, "token_selected must be int32 (T, top_k)")
    top_k = token_selected.shape[1]
    _e4m3(fc1_weights, "fc1_weights"), _e4m3(fc2_weights, "fc2_weights")
    _need(fc1_weights.dim() == 3 and fc1_weights.shape[2] == hdim and
          fc1_weights.shape[1] % 2 == 0, "fc1_weights must be (E, 2 I, H)")
    e, two_i = fc1_weights.shape[0], fc1_weights.shape[1]
    inter = two_i // 2
    _need(tuple(fc2_weights.shape) == (e, hdim, inter), "fc2_weights must be (E, H, I)")
    _need(fc1_scales.dtype == torch.float32 and
          tuple(fc1_scales.shape) == (e, two_i // 128, hdim // 128),
          "fc1_scales must be float32 (E, 2 I / 128, H / 128)")
    _need(fc2_scales.dtype == torch.float32 and
          tuple(fc2_scales.shape) == (e, hdim // 128, inter // 128),
          "fc2_scales must be float32 (E, H / 128, I / 128)")
    _need(out.dtype == torch.bfloat16 and tuple(out.shape) == (t, hdim),
          "out must be bfloat16 (T, H)")
    dev = _cuda_contig((input, token_selected, fc1_weights, fc2_weights, out, fc1_scales,
                        fc2_scales), ("input", "token_selected", "fc1_weights", "fc2_weights",
                                      "out", "fc1_scales", "fc2_scales"))
    return t, e, top_k, hdim, inter, dev


def fused_moe_deepseek_fp8_block_scale(input, token_selected, fc1_weights, fc2_weights, out,
                                       fc1_scales, fc2_scales, workspace=None, stream=None):
    """DeepSeek FP8 block-scale MoE layer (see include/fp8g.h): out (T, H) BF16 =
    sum over each token's selected experts of fc2(SwiGLU(fc1(input))).

    ``workspace`` is a uint8 CUDA tensor of at least ``moe_workspace_size(...)``
    bytes; when omitted one is allocated with torch for this call.
    """
    torch = _torch()
    t, e, top_k, hdim, inter, dev = _moe_args(input, token_selected, fc1_weights, fc2_weights,
                                              out, fc1_scales, fc2_scales)
    need = moe_workspace_size(t, e, top_k, hdim, inter)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _cuda_contig((workspace,), ("workspace",))
    rc = load().fused_moe_deepseek_fp8_block_scale(
        _ptr(input), _ptr(token_selected), _ptr(fc1_weights), _ptr(fc2_weights), _ptr(out),
        _ptr(fc1_scales), _ptr(fc2_scales), t, e, top_k, hdim, inter, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    _raise_on(rc, "fused_moe_deepseek_fp8_block_scale")
    return out


def fused_moe_deepseek_fp8_block_scale_noalloc(input, token_selected, fc1_weights, fc2_weights,
                                               out, fc1_scales, fc2_scales, stream=None):
    """The MoE layer for callers that cannot hand the library device memory (a
    host that reserved all of it for its own pool, a serving loop that must not
    call cudaMalloc): its scratch is the library's fixed per-device array of
    MOE_STATIC_SCRATCH_BYTES and nothing is allocated.  Same checks as the
    workspace form; calls that can overlap on one device race on that array."""
    t, e, top_k, hdim, inter, dev = _moe_args(input, token_selected, fc1_weights, fc2_weights,
                                              out, fc1_scales, fc2_scales)
    rc = load().fused_moe_deepseek_fp8_block_scale_noalloc(
        _ptr(input), _ptr(token_selected), _ptr(fc1_weights), _ptr(fc2_weights), _ptr(out),
        _ptr(fc1_scales), _ptr(fc2_scales), t, e, top_k, hdim, inter,
        _stream_handle(stream, dev))
    _raise_on(rc, "fused_moe_deepseek_fp8_block_scale_noalloc")
    return out


def bmm_fp8(A, B, A_scale, B_scale, dtype=None, out=None, backend="auto", stream=None):
    """The page's ``bmm_fp8``: out (batch, m, n) = A (batch, m, k) @ B (batch, k, n)
    times the scales.  A and B are ``float8_e4m3fn`` or ``float8_e5m2`` (each on its
    own); each scale is a one-element float32 tensor (tensorwise) or channelwise,
    A_scale (batch, m, 1) and B_scale (batch, 1, n).  ``dtype``: bfloat16 or
    float16 output (bfloat16 when omitted; ``out``'s dtype wins)."""
    torch = _torch()
    if backend != "auto":
        raise Fp8gError(ERR_UNSUPPORTED, "bmm_fp8",
                        "only backend='auto' (this library's sm_103a kernel) exists")
    fmts = {torch.float8_e4m3fn: 0, torch.float8_e5m2: 1}
    _need(A.dtype in fmts and B.dtype in fmts, "A and B must be float8_e4m3fn or float8_e5m2")
    _need(A.dim() == 3 and B.dim() == 3, "A must be (batch, m, k) and B (batch, k, n)")
    batch, m, k = A.shape
    n = B.shape[2]
    _need(tuple(B.shape[:2]) == (batch, k), "B must be (%d, %d, n)" % (batch, k))
    a_ch = A_scale.numel() != 1
    b_ch = B_scale.numel() != 1
    _need(A_scale.dtype == torch.float32 and B_scale.dtype == torch.float32,
          "scales must be float32")
    _need(not a_ch or tuple(A_scale.shape) == (batch, m, 1), "channelwise A_scale must be (batch, m, 1)")
    _need(not b_ch or tuple(B_scale.shape) == (batch, 1, n), "channelwise B_scale must be (batch, 1, n)")
    if out is None:
        out = torch.empty((batch, m, n), device=A.device,
                          dtype=dtype if dtype is not None else torch.bfloat16)
    _need(tuple(out.shape) == (batch, m, n), "out must be (batch, m, n)")
    code = _out_code(out.dtype)
    _need(code in (OUT_BF16, OUT_F16), "bmm_fp8 output must be bfloat16 or float16")
    dev = _cuda_contig((A, B, A_scale, B_scale, out), ("A", "B", "A_scale", "B_scale", "out"))
    rc = load().bmm_fp8(_ptr(A), _ptr(B), fmts[A.dtype], fmts[B.dtype], _ptr(A_scale), int(a_ch),
                        _ptr(B_scale), int(b_ch), _ptr(out), code, batch, m, n, k,
                        _stream_handle(stream, dev))
    _raise_on(rc, "bmm_fp8")
    return out


# ------------------------------------------------------------- page signatures

def gemm_fp8_nt_groupwise(a, b, a_scale, b_scale, scale_major_mode=None, mma_sm=None,
                          scale_granularity_mnk=(1, 128, 128), out=None, out_dtype=None,
                          backend="auto", output_scale=None):
    """The page's ``gemm_fp8_nt_groupwise``: returns out (m, n).

    ``mma_sm``: the page's default (1) configures MATE's MUSA kernels; on GB300
    it is a hint, and leaving it out picks the tile shape from the problem size
    (CTA pairs on large problems).  An explicit 1 or 2 forces one SM or a CTA
    pair per tile.  Results are bit-identical either way.
    """
    torch = _torch()
    if backend != "auto":
        raise Fp8gError(ERR_UNSUPPORTED, "gemm_fp8_nt_groupwise",
                        "only backend='auto' (this library's sm_103a kernel) exists")
    _check_granularity(scale_granularity_mnk)
    if out is None:
        default = torch.float8_e4m3fn if output_scale is not None else torch.bfloat16
        out = torch.empty((a.shape[0], b.shape[0]), device=a.device,
                          dtype=out_dtype if out_dtype is not None else default)
    return fp8_gemm_nt_groupwise(a, b, a_scale, b_scale, out, scale_major_mode or "K",
                                 0 if mma_sm is None else mma_sm, scale_granularity_mnk,
                                 output_scale=output_scale)


def group_deepgemm_fp8_nt_groupwise(a, b, a_scale, b_scale, m_indices,
                                    scale_granularity_mnk=(1, 128, 128), out=None,
                                    out_dtype=None):
    """The page's ``group_deepgemm_fp8_nt_groupwise``: returns out (m, n) BF16."""
    torch = _torch()
    _check_granularity(scale_granularity_mnk)
    if out is None:
        if out_dtype not in (None, torch.bfloat16):
            raise TypeError("only bfloat16 output is supported")
        out = torch.empty((a.shape[0], b.shape[1]), device=a.device, dtype=torch.bfloat16)
    return fp8_group_gemm_contiguous(a, b, a_scale, b_scale, m_indices, out)


def batch_deepgemm_fp8_nt_groupwise(a, b, a_scale, b_scale, masked_m, expected_m,
                                    scale_granularity_mnk=(1, 128, 128), out=None,
                                    out_dtype=None):
    """The page's ``batch_deepgemm_fp8_nt_groupwise``: returns out (G, max_m, n) BF16."""
    torch = _torch()
    _check_granularity(scale_granularity_mnk)
    if out is None:
        if out_dtype not in (None, torch.bfloat16):
            raise TypeError("only bfloat16 output is supported")
        out = torch.empty((a.shape[0], a.shape[1], b.shape[1]), device=a.device,
                          dtype=torch.bfloat16)
    return fp8_batch_gemm_masked(a, b, a_scale, b_scale, masked_m, expected_m, out)
