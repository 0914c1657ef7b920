/*
 * fp8g — FP8 (E4M3) groupwise-scaled NT GEMM for sm_103a (GB300).
 *
 * C ABI of the library.  Three GEMMs, as defined on the MATE page
 * "FlashInfer Wrapper APIs", section GEMM, and the kernel that produces their
 * FP8 activations (section Norm, fused_add_rmsnorm_fp8_block_quant, below):
 *
 *   fp8_gemm_nt_groupwise       gemm_fp8_nt_groupwise            out = a @ b.T
 *   fp8_group_gemm_contiguous   group_deepgemm_fp8_nt_groupwise  out[i] = a[i] @ b[m_indices[i]].T
 *   fp8_batch_gemm_masked       batch_deepgemm_fp8_nt_groupwise  out[g,:masked_m[g]] = a[g,:masked_m[g]] @ b[g].T
 *
 * Scaling is groupwise at granularity (1, 128, 128): with KB = k/128,
 *   out[i][j] = sum_kb ( sum_{t in block kb} a[i][t] * b[j][t] ) * a_scale(i, kb) * b_scale(j/128, kb)
 * where a and b hold E4M3 (float8_e4m3fn) codes and the scales are FP32
 * multipliers (dequantisation factors).  Block sums are accumulated in FP32 on
 * the tensor cores, scaled and summed in FP32, and rounded once to the output
 * type (round to nearest even).
 *
 * Conventions, shared by every entry point (the ownership and error model of
 * the "flashmla-rs" page, section Design Notes, and the asynchronous calls of
 * the "flashinfer-rs" page, section Additional Notes):
 *   - All array arguments are DEVICE pointers owned by the caller.  The
 *     library allocates nothing per call and keeps no pointer after return.
 *   - Work is enqueued on `stream` and the call returns without synchronising.
 *     Results are ready when the stream reaches that point.
 *   - Every argument is checked on the host before anything is launched; a
 *     rejected call launches nothing and leaves `out` untouched.  No C++
 *     exception crosses the ABI.  On failure the return value says why and
 *     fp8g_last_error() gives a message.
 *   - Device requirements: compute capability 10.3 (sm_103, GB300), else
 *     FP8G_ERR_ARCH.
 *   - Shapes: k and n must be positive multiples of 128 (the scale
 *     granularity); m (and max_m, M_total) may be any non-negative value,
 *     including 0 (nothing is launched).  Every dimension must be < 2^31.
 *   - Alignment: a, b and out 16-byte aligned; scales 4-byte aligned;
 *     m_indices / masked_m 4-byte aligned.  All arrays densely packed
 *     (contiguous, row-major, no padding between rows).
 *   - Calls are thread-safe.  Calls on different streams may run concurrently.
 */
#ifndef FP8G_H
#define FP8G_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8G_OK = 0,
    FP8G_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad shape, misalignment, bad enum */
    FP8G_ERR_UNSUPPORTED = 2,      /* valid on the page but not provided here */
    FP8G_ERR_ARCH = 3,             /* current device is not sm_103 */
    FP8G_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed */
    FP8G_ERR_TIMEOUT = 5           /* reported through the device status word */
} fp8g_status_t;

/* Scale layout of the dense form (page: scale_major_mode; None means "K").
 *   K-major:  a_scale (m, k/128),   b_scale (n/128, k/128)
 *   MN-major: a_scale (k/128, m),   b_scale (k/128, n/128)              */
typedef enum { FP8G_SCALE_K_MAJOR = 0, FP8G_SCALE_MN_MAJOR = 1 } fp8g_scale_major_t;

/* Output element type: BF16 (the page's default), FP16, or E4M3 codes with a
 * per-tensor FP32 output scale (the page's output_scale path). */
typedef enum { FP8G_OUT_BF16 = 0, FP8G_OUT_F16 = 1, FP8G_OUT_E4M3 = 2 } fp8g_dtype_t;

/* FP8 formats of bmm_fp8's operands. */
typedef enum { FP8G_FP8_E4M3 = 0, FP8G_FP8_E5M2 = 1 } fp8g_fp8_format_t;

/* Bits of the device status word (see fp8g_get_device_status). */
#define FP8G_DEVICE_TIMEOUT 0x1u          /* a pipeline wait exceeded its limit; the launch gave up */
#define FP8G_DEVICE_BAD_M_INDICES 0x2u    /* a 128-row block broke the contiguous-layout precondition; skipped */
#define FP8G_DEVICE_MASKED_M_CLAMPED 0x4u /* some masked_m[g] was outside [0, max_m]; clamped */

/*
 * Dense groupwise FP8 NT GEMM (page: gemm_fp8_nt_groupwise).
 *
 *   a        (m, k)  E4M3 codes, row-major.
 *   b        (n, k)  E4M3 codes, row-major; the operation is a @ b.T.
 *   a_scale  FP32, (m, k/128) if K-major, (k/128, m) if MN-major.
 *   b_scale  FP32, (n/128, k/128) if K-major, (k/128, n/128) if MN-major.
 *   out      (m, n) row-major, BF16, FP16 or E4M3 per out_dtype.  Every
 *            element is written.
 *   output_scale  NULL for BF16/FP16 output.  For FP8G_OUT_E4M3 (and only
 *            then) a device pointer to one FP32 value s > 0, the scale of the
 *            FP8 output in the same sense as a_scale and b_scale (value =
 *            code * s): out = E4M3(R * (1/s)) with R the FP32 result, 1/s
 *            correctly rounded, round to nearest even, saturated to +-448.
 *   gran_m, gran_n, gran_k   the page's scale_granularity_mnk; only
 *            (1, 128, 128) is provided, anything else is FP8G_ERR_UNSUPPORTED.
 *   mma_sm   the page's MMA configuration hint: 0 (auto), 1 or 2.  It may
 *            change speed, never results.
 */
fp8g_status_t fp8_gemm_nt_groupwise(const void* a, const void* b,
                                    const float* a_scale, const float* b_scale,
                                    void* out, fp8g_dtype_t out_dtype,
                                    const float* output_scale,
                                    int64_t m, int64_t n, int64_t k,
                                    fp8g_scale_major_t scale_major,
                                    int gran_m, int gran_n, int gran_k,
                                    int mma_sm, cudaStream_t stream);

/*
 * Batched FP8 GEMM with tensorwise or channelwise scales (page: bmm_fp8).
 *
 *   a        (batch, m, k) FP8 codes, row-major; format a_format (E4M3 or E5M2).
 *   b        (batch, k, n) FP8 codes, row-major; format b_format.  The operation
 *            is a[b] @ b[b] (B is not transposed, unlike the NT forms above).
 *   a_scale  FP32: one value (a_channelwise == 0) or (batch, m, 1), one per row of a.
 *   b_scale  FP32: one value (b_channelwise == 0) or (batch, 1, n), one per column of b.
 *   out      (batch, m, n) row-major, BF16 or FP16; every element is written.
 *
 *   out[b][i][j] = round( (sum_t a[b][i][t] * b[b][t][j]) * a_scale(b, i) * b_scale(b, j) )
 *
 * The sum over k is accumulated in FP32 on the tensor cores (no per-block
 * promotion is needed, as the scales do not depend on k) and scaled once.
 * n and k must be positive multiples of 16 (TMA reads rows whose pitch is a
 * multiple of 16 bytes; the page states no constraint); batch and m may be 0.
 * a, b, out 16-byte aligned, scales 4-byte aligned.  Otherwise
 * FP8G_ERR_INVALID_ARGUMENT, nothing launched.
 */
fp8g_status_t bmm_fp8(const void* a, const void* b, fp8g_fp8_format_t a_format,
                      fp8g_fp8_format_t b_format, const float* a_scale, int a_channelwise,
                      const float* b_scale, int b_channelwise, void* out,
                      fp8g_dtype_t out_dtype, int64_t batch, int64_t m, int64_t n, int64_t k,
                      cudaStream_t stream);

/*
 * Contiguous grouped FP8 NT GEMM for MoE experts
 * (page: group_deepgemm_fp8_nt_groupwise).
 *
 *   a          (m, k) E4M3, the rows of all experts stacked (m = M_total).
 *   b          (num_groups, n, k) E4M3 expert weights.
 *   a_scale    FP32 (m, k/128), K-major.
 *   b_scale    FP32 (num_groups, n/128, k/128), K-major.
 *   m_indices  int32 (m): the expert of each row, -1 for a padding row.
 *              Precondition (page): each expert's rows occupy a contiguous
 *              region starting on a multiple of 128 rows, so every 128-row
 *              block holds rows of at most one expert plus -1 padding.
 *   out        (m, n) BF16.  Rows with m_indices == -1 are not written (the
 *              page leaves them unspecified).
 *   A block that breaks the precondition (an id outside [-1, num_groups) or
 *   two experts in one block) is skipped, not written, and raises
 *   FP8G_DEVICE_BAD_M_INDICES in the device status word; it never faults.
 */
fp8g_status_t fp8_group_gemm_contiguous(const void* a, const void* b,
                                        const float* a_scale, const float* b_scale,
                                        const int32_t* m_indices, void* out,
                                        int64_t m, int64_t n, int64_t k,
                                        int64_t num_groups, cudaStream_t stream);

/*
 * Masked batched FP8 NT GEMM for MoE decode
 * (page: batch_deepgemm_fp8_nt_groupwise).
 *
 *   a          (num_groups, max_m, k) E4M3.
 *   b          (num_groups, n, k) E4M3.
 *   a_scale    FP32 (num_groups, max_m, k/128), K-major.
 *   b_scale    FP32 (num_groups, n/128, k/128), K-major.
 *   masked_m   int32 (num_groups), device memory: valid rows per group.
 *              Values outside [0, max_m] are clamped and raise
 *              FP8G_DEVICE_MASKED_M_CLAMPED.
 *   expected_m the page's host-side row-count hint (>= 0).  It may change
 *              speed, never results.
 *   out        (num_groups, max_m, n) BF16.  Rows at or beyond masked_m[g] are
 *              not written (the page leaves them unspecified).
 */
fp8g_status_t fp8_batch_gemm_masked(const void* a, const void* b,
                                    const float* a_scale, const float* b_scale,
                                    const int32_t* masked_m, int64_t expected_m,
                                    void* out, int64_t num_groups, int64_t max_m,
                                    int64_t n, int64_t k, cudaStream_t stream);

/*
 * Fused add + RMSNorm + row-major 1 x 128 FP8 quantisation, the producer of the
 * GEMMs' `a` and K-major `a_scale` (page: fused_add_rmsnorm_fp8_block_quant,
 * section Norm).  Per row of `hidden` BF16 values:
 *
 *   residual_j   <- BF16(input_j + residual_j)                 (in place)
 *   normed_out_j  = BF16(residual_j * r * weight_j),  r = 1 / sqrt(mean(residual^2) + eps)
 *   for every 128-column block b:
 *     block_scale[b] = amax_b / 448 (FP32), amax_b = max over the block of |normed_out_j|
 *     out_j          = E4M3(normed_out_j / block_scale[b]), round to nearest even,
 *                      saturated to +-448; an all-zero block gets scale 0, codes 0
 *
 * so that normed_out_j ~= out_j * block_scale[b] (the scales are multipliers,
 * as the GEMMs' a_scale).
 *
 *   out          (rows, hidden) E4M3 codes.
 *   block_scale  FP32 (rows, hidden/128), row-major (the GEMMs' K-major a_scale).
 *   normed_out   (rows, hidden) BF16.
 *   input        (rows, hidden) BF16, read only.
 *   residual     (rows, hidden) BF16, read and overwritten with input + residual.
 *   weight       (hidden) BF16.
 *   eps          added to the mean square (page default 1e-6), >= 0.
 *   hidden must be a positive multiple of 128 and at most 65536; rows >= 0
 *   (0 launches nothing).  out, normed_out, input, residual and weight 16-byte
 *   aligned, block_scale 4-byte aligned; the arrays must not overlap.
 *   Accumulation is FP32, so normed_out may differ from an exact computation
 *   by one BF16 unit in the last place where the exact value is close to a
 *   rounding boundary; the codes and scales are a deterministic function of
 *   normed_out.
 */
fp8g_status_t fused_add_rmsnorm_fp8_block_quant(void* out, float* block_scale, void* normed_out,
                                                const void* input, void* residual,
                                                const void* weight, float eps, int64_t rows,
                                                int64_t hidden, cudaStream_t stream);

/*
 * DeepSeek FP8 block-scale MoE layer ("flashinfer-rs" page, section "API
 * Example: Fused MoE FP8 (cudarc)", fused_moe_cudarc_deepseek_fp8_block_scale),
 * built on fp8_group_gemm_contiguous.  With T = num_tokens, K = top_k,
 * E = num_experts, H = hidden_size, I = inter_size, for every token t:
 *
 *   (xq, xs) = 1x128 E4M3 quantisation of input[t]   (scale = amax / 448, as in
 *                                                     fused_add_rmsnorm_fp8_block_quant)
 *   for each slot s with e = token_selected[t, s] != -1:
 *     h   = BF16(fc1_e(xq, xs))     rows [0, I) of h are the gate, [I, 2 I) the up part
 *     act = silu(h[0:I]) * h[I:2I]  (FP32; silu with the hardware exponential and
 *                                    divide), then its 1x128 quantisation
 *     y   = BF16(fc2_e(act))
 *   out[t] = BF16(sum of y over the token's slots)   (no routing weights: the
 *                                                     page's signature has none)
 *
 * where fc(x)_j = sum_kb blocksum * x_scale[kb] * w_scale[j/128][kb] as in the GEMMs.
 *
 *   input           (T, H) BF16.
 *   token_selected  (T, K) int32 expert ids in [0, E), -1 for an empty slot.  Any
 *                   other value is skipped and raises FP8G_DEVICE_BAD_M_INDICES.
 *   fc1_weights     (E, 2 I, H) E4M3;  fc1_scales (E, 2 I / 128, H / 128) FP32.
 *   fc2_weights     (E, H, I) E4M3;    fc2_scales (E, H / 128, I / 128) FP32.
 *   out             (T, H) BF16; every element is written (zeros for a token
 *                   without a valid slot).
 *   workspace       caller-owned device scratch of at least
 *                   fused_moe_deepseek_fp8_block_scale_workspace_size(...) bytes,
 *                   256-byte aligned; its contents on entry do not matter.  Two
 *                   calls must not share a workspace while both may be running.
 *   H and I must be positive multiples of 128, 1 <= K <= E <= 4096, T >= 0 (0
 *   launches nothing).  input, weights and out 16-byte aligned, token_selected
 *   and scales 4-byte aligned.
 */
size_t fused_moe_deepseek_fp8_block_scale_workspace_size(int64_t num_tokens, int64_t num_experts,
                                                         int64_t top_k, int64_t hidden_size,
                                                         int64_t inter_size);
fp8g_status_t fused_moe_deepseek_fp8_block_scale(
    const void* input, const int32_t* token_selected, const void* fc1_weights,
    const void* fc2_weights, void* out, const float* fc1_scales, const float* fc2_scales,
    int64_t num_tokens, int64_t num_experts, int64_t top_k, int64_t hidden_size,
    int64_t inter_size, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The MoE layer above without a caller workspace.  The pages have no
 * counterpart of this call.  It is for callers that have no way to give the
 * library device memory: a host program that hands all of the GPU's memory to
 * its own pool at start-up and offers a plug-in no allocator, or a serving loop
 * that must never call cudaMalloc because that call can wait for the whole
 * device and stall every stream.  Such a caller still passes its inputs and
 * output; the layer's scratch lives in a fixed array of
 * FP8G_MOE_STATIC_SCRATCH_BYTES that the library defines statically, and the
 * call allocates nothing (no cudaMalloc, no cudaFree, no allocating library).
 *
 *   - Cost: every device on which the library's kernels are loaded holds this
 *     array from then until the process exits, whether or not the call is used.
 *   - Set-up: the first call on a device looks the array's device address up
 *     (a host-side query, once per device, under a lock).  Make that first call
 *     on each device before any stream capture begins.
 *   - Problems whose scratch (fused_moe_deepseek_fp8_block_scale_workspace_size)
 *     exceeds FP8G_MOE_STATIC_SCRATCH_BYTES return FP8G_ERR_UNSUPPORTED with a
 *     message giving both sizes; nothing is launched.
 *   - Nothing in the scratch has to start at zero: the routing step writes every
 *     entry of the layout it reads back, and every other region is written
 *     before it is read within the same call.  The array keeps the last call's
 *     intermediates (layout as in ..._workspace_layout).
 *   - There is one array per device: calls that may run at the same time on
 *     one device (different streams, or host threads) race on it and corrupt
 *     each other's results.  Calls in one stream are ordered and safe.
 */
#define FP8G_MOE_STATIC_SCRATCH_BYTES (64u << 20) /* 64 MiB */
fp8g_status_t fused_moe_deepseek_fp8_block_scale_noalloc(
    const void* input, const int32_t* token_selected, const void* fc1_weights,
    const void* fc2_weights, void* out, const float* fc1_scales, const float* fc2_scales,
    int64_t num_tokens, int64_t num_experts, int64_t top_k, int64_t hidden_size,
    int64_t inter_size, cudaStream_t stream);

/*
 * Layout of the MoE layer's workspace (the same layout sits in the static
 * scratch of the allocation-free entry point).  Writes the number of rows M of
 * the routed layout to *rows and the byte offsets of its eight regions, each
 * 256-byte aligned, to offsets[0..7]:
 *   0 m_indices  int32 (M)              expert of each routed row, -1 = padding
 *   1 row_of     int32 (T, K)           routed row of each slot, -1 = empty slot
 *   2 a1         E4M3 (M, H)            quantised input rows
 *   3 a1_scale   FP32 (M, H / 128)      their 1x128 scales
 *   4 h          BF16 (M, 2 I)          fc1 output (gate, then up)
 *   5 a2         E4M3 (M, I)            quantised SwiGLU activations
 *   6 a2_scale   FP32 (M, I / 128)      their 1x128 scales
 *   7 y          BF16 (M, H)            fc2 output
 * with M = round_up(T * K + 127 * E, 128).  After a call, the regions hold that
 * call's intermediates on the rows m_indices marks as routed (other rows are
 * unspecified); the row order inside an expert's segment may differ from call
 * to call.  Same argument checks as the workspace size query.
 */
fp8g_status_t fused_moe_deepseek_fp8_block_scale_workspace_layout(
    int64_t num_tokens, int64_t num_experts, int64_t top_k, int64_t hidden_size,
    int64_t inter_size, int64_t* rows, size_t offsets[8]);

/* Message of the last failed call on this thread ("" if none); valid until the
 * thread's next call into the library. */
const char* fp8g_last_error(void);

/*
 * Device status word of the current device: an OR of FP8G_DEVICE_* bits set by
 * kernels since it was last cleared.  Synchronises the device first, then
 * copies the word to *flags and, if `clear` is non-zero, resets it.  Returns
 * FP8G_ERR_TIMEOUT if the timeout bit is set, FP8G_OK otherwise (other bits
 * are reported through *flags only).
 */
fp8g_status_t fp8g_get_device_status(unsigned int* flags, int clear);

/*
 * The same word, read in the order of `stream`: waits for the work enqueued on
 * `stream` so far (and only that stream), copies the word to *flags and, if
 * `clear` is non-zero, resets it, both as steps of the stream.  The word is
 * shared by every stream of the device, so it also holds bits that kernels on
 * other streams have raised by then.  Same return values as
 * fp8g_get_device_status.
 */
fp8g_status_t fp8g_get_stream_status(unsigned int* flags, int clear, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8G_H */
