/*
 * CPU oracle for the FP8 (E4M3) groupwise-scaled NT GEMM and its two MoE forms.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes is the plain definition of the operations on the MATE page
 * "FlashInfer Wrapper APIs", section GEMM (and, for the producer of the GEMM's
 * FP8 activations, section Norm, declared further down):
 *   - gemm_fp8_nt_groupwise:            out = a @ b.T with FP32 scales at
 *                                       granularity (1, 128, 128)
 *   - group_deepgemm_fp8_nt_groupwise:  out[i] = a[i] @ b[m_indices[i]].T
 *   - batch_deepgemm_fp8_nt_groupwise:  out[g, :masked_m[g]] =
 *                                       a[g, :masked_m[g]] @ b[g].T
 *
 * With dec() the E4M3 decode, KB = k/128 and sa/sb the scales:
 *   P(i,j,kb) = sum_{t in block kb} dec(a[i,t]) * dec(b[j,t])          (FP64)
 *   R(i,j)    = sum_kb P(i,j,kb) * ((double)sa(i,kb) * (double)sb(j/128,kb))
 *   out(i,j)  = R(i,j) rounded once, to nearest even, to BF16 or FP16.
 *
 * Each block sum P is exact in FP64 (every E4M3 value is an integer multiple
 * of 2^-9 no larger than 448, so a 128-term sum of products needs < 44
 * significant bits), and so is the scale product (24 + 24 bits).  The only
 * roundings are the FP64 sum over K blocks and the final conversion.
 *
 * Every function returns 0 on success and a negative value if its arguments
 * violate a precondition of the page (bad shape, m_indices outside [-1, G),
 * an expert id that changes inside a 128-row block).
 */
#ifndef FP8G_ORACLE_H
#define FP8G_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Output formats of the final rounding. */
#define ORACLE_OUT_BF16 0
#define ORACLE_OUT_F16 1

/* Scale layouts: K-major a_scale (m, k/128), b_scale (n/128, k/128);
 * MN-major a_scale (k/128, m), b_scale (k/128, n/128). */
#define ORACLE_SCALE_K_MAJOR 0
#define ORACLE_SCALE_MN_MAJOR 1

/* The 256-entry E4M3 (float8_e4m3fn) decode table, built from the format
 * definition: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, exponent 1111 with mantissa 111 is NaN. */
void oracle_e4m3_table(double out[256]);

/* Round x once, to nearest with ties to even, to BF16 or FP16.  Writes the
 * rounded value (as a double) and its 16-bit encoding.  Overflow gives +-inf
 * under the usual round-to-nearest rule, NaN stays NaN. */
void oracle_round(const double* x, int64_t count, int out_dtype,
                  double* rounded, uint16_t* bits);

/* Dense form.  a (m,k) and b (n,k) are row-major E4M3 codes.  ref (m*n) gets
 * R before rounding, out (m*n) the rounded 16-bit codes; either may be NULL. */
int oracle_gemm_nt_groupwise(const uint8_t* a, const uint8_t* b,
                             const float* a_scale, const float* b_scale,
                             int64_t m, int64_t n, int64_t k, int scale_major,
                             int out_dtype, double* ref, uint16_t* out);

/* Dense form at `count` chosen positions (rows[s], cols[s]); ref/out have
 * `count` entries. */
int oracle_gemm_nt_groupwise_at(const uint8_t* a, const uint8_t* b,
                                const float* a_scale, const float* b_scale,
                                int64_t m, int64_t n, int64_t k, int scale_major,
                                int out_dtype, const int64_t* rows,
                                const int64_t* cols, int64_t count,
                                double* ref, uint16_t* out);

/* Contiguous grouped form.  a (m,k), b (G,n,k), a_scale (m,k/128) and
 * b_scale (G,n/128,k/128), all K-major; m_indices (m) with -1 for padding.
 * Rows with m_indices == -1 are not computed: written[i] = 0 there and 1
 * elsewhere (written may be NULL), and ref/out rows are left untouched. */
int oracle_group_gemm_contiguous(const uint8_t* a, const uint8_t* b,
                                 const float* a_scale, const float* b_scale,
                                 const int32_t* m_indices, int64_t m, int64_t n,
                                 int64_t k, int64_t num_groups, double* ref,
                                 uint16_t* out, uint8_t* written);

/* Grouped form at chosen positions; a position on a padding row gets
 * written[s] = 0 and is left untouched. */
int oracle_group_gemm_contiguous_at(const uint8_t* a, const uint8_t* b,
                                    const float* a_scale, const float* b_scale,
                                    const int32_t* m_indices, int64_t m,
                                    int64_t n, int64_t k, int64_t num_groups,
                                    const int64_t* rows, const int64_t* cols,
                                    int64_t count, double* ref, uint16_t* out,
                                    uint8_t* written);

/* Masked batched form.  a (G,max_m,k), b (G,n,k), a_scale (G,max_m,k/128),
 * b_scale (G,n/128,k/128); masked_m (G).  Row r of group g is computed when
 * r < clamp(masked_m[g], 0, max_m); other rows are left untouched and get
 * written = 0.  Indices into ref/out/written are g*max_m*n + r*n + j. */
int oracle_batch_gemm_masked(const uint8_t* a, const uint8_t* b,
                             const float* a_scale, const float* b_scale,
                             const int32_t* masked_m, int64_t num_groups,
                             int64_t max_m, int64_t n, int64_t k, double* ref,
                             uint16_t* out, uint8_t* written);

/* Masked form at chosen positions: groups[s], rows[s] (row within the group)
 * and cols[s]. */
int oracle_batch_gemm_masked_at(const uint8_t* a, const uint8_t* b,
                                const float* a_scale, const float* b_scale,
                                const int32_t* masked_m, int64_t num_groups,
                                int64_t max_m, int64_t n, int64_t k,
                                const int64_t* groups, const int64_t* rows,
                                const int64_t* cols, int64_t count, double* ref,
                                uint16_t* out, uint8_t* written);

/* Encode values as E4M3 codes (float8_e4m3fn): round to nearest with ties to
 * even on the format's grid (3 mantissa bits, subnormal quantum 2^-9) and
 * saturate to +-448 (the format has no infinity); NaN gives 0x7F. */
void oracle_e4m3_encode(const double* x, int64_t count, uint8_t* codes);

/* fused_add_rmsnorm_fp8_block_quant of the MATE page "FlashInfer Wrapper
 * APIs", section Norm: add `input` to `residual`, RMS-normalise the sum and
 * quantise it to FP8 E4M3 with one FP32 scale per row-major 1 x 128 block.
 * All BF16 tensors are passed as their 16-bit encodings; input, residual,
 * residual_out and normed_out are (rows, hidden), weight is (hidden), out is
 * (rows, hidden) E4M3 codes, block_scale is (rows, hidden / 128).  Per row:
 *   x_j      = BF16(input_j + residual_j)                 -> residual_out
 *   r        = 1 / sqrt(sum_j x_j^2 / hidden + eps)       (FP64)
 *   y_j      = BF16(x_j * r * weight_j)                   -> normed_out
 *   per block: amax = max |y_j|, scale = FP32(amax / 448) -> block_scale
 *              code_j = E4M3(FP32(y_j / scale))           -> out
 * (an all-zero block gets scale 0 and codes 0).  Returns -1 unless hidden is a
 * positive multiple of 128 and rows >= 0. */
int oracle_fused_add_rmsnorm_fp8_block_quant(const uint16_t* input,
                                             const uint16_t* residual,
                                             const uint16_t* weight, double eps,
                                             int64_t rows, int64_t hidden,
                                             uint16_t* residual_out,
                                             uint16_t* normed_out, uint8_t* out,
                                             float* block_scale);

/* Row-major 1 x 128 FP8 quantisation of FP64 values (rows, cols), cols a
 * multiple of 128: per block scale = FP32(amax / 448), code = E4M3(FP32(x /
 * scale)); an all-zero block gets scale 0 and codes 0.  codes (rows, cols),
 * scales (rows, cols / 128). */
void oracle_quant_1x128(const double* x, int64_t rows, int64_t cols, uint8_t* codes,
                        float* scales);

/* The DeepSeek FP8 block-scale MoE layer of the "flashinfer-rs" page, section
 * "API Example: Fused MoE FP8 (cudarc)", DeepSeek FP8 block-scale mode, built
 * from the groupwise GEMM of the MATE page, section GEMM.  For every token t:
 *   (xq, xs) = 1x128 quantisation of input[t]                (BF16 -> E4M3)
 *   for each of its top_k slots with expert e = token_selected[t, s] >= 0:
 *     h   = BF16(fc1_e(xq))     fc1 (E, 2*inter, hidden) E4M3, scales s1
 *                               (E, 2*inter/128, hidden/128); rows [0, inter)
 *                               of h are the gate, [inter, 2*inter) the up part
 *     act = silu(h_gate) * h_up                              (FP64)
 *     (aq, as) = 1x128 quantisation of act
 *     y   = BF16(fc2_e(aq))     fc2 (E, hidden, inter) E4M3, scales s2
 *                               (E, hidden/128, inter/128)
 *   out[t] = BF16(sum of y over the token's slots)           (unweighted)
 * with fc(x)_j = sum_kb (block sum) * x_scale[kb] * w_scale[j/128][kb] as in the
 * GEMM.  input and out are BF16 encodings (tokens, hidden); token_selected is
 * (tokens, top_k) with -1 for an empty slot.  Returns -1 on a bad shape, -2 if
 * an expert id lies outside [-1, num_experts). */
int oracle_moe_deepseek_fp8_block_scale(const uint16_t* input, const int32_t* token_selected,
                                        const uint8_t* w1, const uint8_t* w2,
                                        const float* s1, const float* s2, int64_t num_tokens,
                                        int64_t num_experts, int64_t top_k, int64_t hidden,
                                        int64_t inter, uint16_t* out);

/* The SwiGLU step of the MoE layer above on given fc1 outputs: for each of
 * `rows` rows of h (BF16 encodings, 2*inter wide: gate, then up),
 * act = silu(gate) * up in FP64 and its 1x128 quantisation, codes (rows, inter)
 * and scales (rows, inter/128) -- the same function the layer applies.
 * Returns -1 unless inter is a positive multiple of 128 and rows >= 0. */
int oracle_moe_swiglu_quant(const uint16_t* h, int64_t rows, int64_t inter, uint8_t* codes,
                            float* scales);

/* The combine step of the MoE layer above on given fc2 outputs: out[t] =
 * BF16(sum over the slots s with row_of[t, s] >= 0 of y[row_of[t, s]]), the
 * sum exact in FP64 and rounded once; y (rows, hidden) and out (tokens, hidden)
 * are BF16 encodings, row_of (tokens, top_k). */
int oracle_moe_combine(const uint16_t* y, const int32_t* row_of, int64_t tokens, int64_t top_k,
                       int64_t hidden, uint16_t* out);

/* FP8 formats of bmm_fp8's operands. */
#define ORACLE_FP8_E4M3 0
#define ORACLE_FP8_E5M2 1

/* The 256-entry E5M2 (float8_e5m2) decode table: 1 sign bit, 5 exponent bits
 * with bias 15, 2 mantissa bits; exponent 11111 is infinity (mantissa 0) or
 * NaN. */
void oracle_e5m2_table(double out[256]);

/* bmm_fp8 of the MATE page "FlashInfer Wrapper APIs", section GEMM: for each
 * batch bb, out[bb] = (A[bb] @ B[bb]) * a_scale * b_scale with A (batch, m, k)
 * and B (batch, k, n) row-major FP8 codes (E4M3 or E5M2 each, a_fmt / b_fmt),
 * and FP32 scales that are either one tensorwise value or channelwise: a_scale
 * (batch, m, 1) per row of A, b_scale (batch, 1, n) per column of B.
 *   out[bb][i][j] = round( (sum_t A[bb][i][t] * B[bb][t][j]) * (sa * sb) )
 * summed in FP64, rounded once to BF16/FP16.  ref/out (batch*m*n), either may
 * be NULL. */
int oracle_bmm_fp8(const uint8_t* a, const uint8_t* b, int a_fmt, int b_fmt,
                   const float* a_scale, int a_channelwise, const float* b_scale,
                   int b_channelwise, int64_t batch, int64_t m, int64_t n, int64_t k,
                   int out_dtype, double* ref, uint16_t* out);

/* Number of threads the oracle's parallel loops use. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif

#endif
