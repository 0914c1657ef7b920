/*
 * CPU oracle for the FP8 (E4M3) groupwise-scaled NT GEMM — TEST INFRASTRUCTURE.
 *
 * Plain, slow and written to be checked by eye against the definition on the
 * MATE page "FlashInfer Wrapper APIs", section GEMM (gemm_fp8_nt_groupwise,
 * group_deepgemm_fp8_nt_groupwise, batch_deepgemm_fp8_nt_groupwise).  No
 * blocking, no reordering: one output element at a time, one 128-wide K block
 * at a time, in FP64, then one rounding.  The only parallelism is over output
 * elements, which does not change any arithmetic.
 *
 * Built with -ffp-contract=off so that no multiply-add is fused and the
 * results are the same on every host.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define KBLOCK 128 /* scale granularity along k, (1, 128, 128) */
#define NBLOCK 128 /* scale granularity along n */

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* E4M3 as named by the page (torch.float8_e4m3fn): sign s, exponent field e
 * (bias 7), mantissa field f.  e == 0 is subnormal: f * 2^-3 * 2^(1-7).
 * Otherwise (1 + f/8) * 2^(e-7).  e == 15 with f == 7 is NaN; there is no
 * infinity, so e == 15 with f < 7 are ordinary finite values (max 448). */
void oracle_e4m3_table(double out[256])
{
    for (int c = 0; c < 256; ++c) {
        int s = (c >> 7) & 1;
        int e = (c >> 3) & 15;
        int f = c & 7;
        double v;
        if (e == 15 && f == 7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)f, -9);
        else
            v = ldexp((double)(8 + f), e - 10);
        out[c] = s ? -v : v;
    }
}

/* Round to nearest, ties to even, into a binary format with p significand
 * bits (including the implicit one), smallest normal exponent emin and
 * largest finite value maxfinite.  The rounding quantum is 2^(E - p + 1) with
 * E the exponent of the leading bit of |x| (floored at emin for subnormals);
 * dividing by it is exact, nearbyint() rounds to even in the default mode. */
static double round_to_format(double x, int p, int emin, double maxfinite)
{
    if (isnan(x) || isinf(x) || x == 0.0)
        return x;
    int e2;
    frexp(fabs(x), &e2); /* |x| = f * 2^e2, f in [0.5, 1) */
    int lead = e2 - 1;
    if (lead < emin)
        lead = emin;
    double quantum = ldexp(1.0, lead - (p - 1));
    double y = nearbyint(x / quantum) * quantum;
    if (fabs(y) > maxfinite)
        return copysign(INFINITY, x);
    return y;
}

#define BF16_P 8
#define BF16_EMIN (-126)
#define BF16_MAX 3.3895313892515355e38 /* (2 - 2^-7) * 2^127 */
#define F16_P 11
#define F16_EMIN (-14)
#define F16_MAX 65504.0

/* 16-bit encodings of a value that is already representable in the format. */
static uint16_t encode_bf16(double y)
{
    if (isnan(y))
        return (uint16_t)0x7FC0;
    union {
        float f;
        uint32_t u;
    } v;
    v.f = (float)y; /* exact: every BF16 value is an FP32 value */
    return (uint16_t)(v.u >> 16);
}

static uint16_t encode_f16(double y)
{
    if (isnan(y))
        return (uint16_t)0x7E00;
    uint16_t sign = signbit(y) ? 0x8000 : 0;
    double a = fabs(y);
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00);
    if (a == 0.0)
        return sign;
    if (a < ldexp(1.0, F16_EMIN)) /* subnormal: a = mant * 2^-24 */
        return (uint16_t)(sign | (uint16_t)ldexp(a, 24));
    int e2;
    frexp(a, &e2);
    int lead = e2 - 1; /* a = (1 + mant/1024) * 2^lead */
    uint16_t mant = (uint16_t)(ldexp(a, 10 - lead) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((lead + 15) << 10) | mant);
}

static double round_one(double x, int out_dtype, uint16_t* bits)
{
    double y;
    if (out_dtype == ORACLE_OUT_F16) {
        y = round_to_format(x, F16_P, F16_EMIN, F16_MAX);
        if (bits)
            *bits = encode_f16(y);
    } else {
        y = round_to_format(x, BF16_P, BF16_EMIN, BF16_MAX);
        if (bits)
            *bits = encode_bf16(y);
    }
    return y;
}

void oracle_round(const double* x, int64_t count, int out_dtype,
                  double* rounded, uint16_t* bits)
{
    for (int64_t s = 0; s < count; ++s) {
        double y = round_one(x[s], out_dtype, bits ? bits + s : NULL);
        if (rounded)
            rounded[s] = y;
    }
}

/* One output element of the definition.  arow/brow are the k codes of row i
 * of a and row j of b; sa[kb*sa_step] and sb[kb*sb_step] are the scales of
 * K block kb for that row of a and that 128-column block of b. */
static double element(const double* dec, const uint8_t* arow,
                      const uint8_t* brow, const float* sa, int64_t sa_step,
                      const float* sb, int64_t sb_step, int64_t kblocks)
{
    double r = 0.0;
    for (int64_t kb = 0; kb < kblocks; ++kb) {
        double p = 0.0; /* exact block sum */
        for (int64_t t = kb * KBLOCK; t < (kb + 1) * KBLOCK; ++t)
            p += dec[arow[t]] * dec[brow[t]];
        double scale = (double)sa[kb * sa_step] * (double)sb[kb * sb_step];
        r += p * scale;
    }
    return r;
}

static int check_dense_shape(int64_t m, int64_t n, int64_t k, int scale_major,
                             int out_dtype)
{
    if (m < 0 || n <= 0 || k <= 0 || n % NBLOCK || k % KBLOCK)
        return -1;
    if (scale_major != ORACLE_SCALE_K_MAJOR &&
        scale_major != ORACLE_SCALE_MN_MAJOR)
        return -1;
    if (out_dtype != ORACLE_OUT_BF16 && out_dtype != ORACLE_OUT_F16)
        return -1;
    return 0;
}

/* Dense element (i, j) with the scale layout of the page: K-major
 * a_scale[i][kb], b_scale[j/128][kb]; MN-major a_scale[kb][i],
 * b_scale[kb][j/128]. */
static double dense_element(const double* dec, const uint8_t* a,
                            const uint8_t* b, const float* a_scale,
                            const float* b_scale, int64_t m, int64_t n,
                            int64_t k, int scale_major, int64_t i, int64_t j)
{
    int64_t kblocks = k / KBLOCK, nblocks = n / NBLOCK, jb = j / NBLOCK;
    const float *sa, *sb;
    int64_t sa_step, sb_step;
    if (scale_major == ORACLE_SCALE_K_MAJOR) {
        sa = a_scale + i * kblocks;
        sa_step = 1;
        sb = b_scale + jb * kblocks;
        sb_step = 1;
    } else {
        sa = a_scale + i;
        sa_step = m;
        sb = b_scale + jb;
        sb_step = nblocks;
    }
    return element(dec, a + i * k, b + j * k, sa, sa_step, sb, sb_step,
                   kblocks);
}

int oracle_gemm_nt_groupwise(const uint8_t* a, const uint8_t* b,
                             const float* a_scale, const float* b_scale,
                             int64_t m, int64_t n, int64_t k, int scale_major,
                             int out_dtype, double* ref, uint16_t* out)
{
    if (check_dense_shape(m, n, k, scale_major, out_dtype))
        return -1;
    double dec[256];
    oracle_e4m3_table(dec);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double r = dense_element(dec, a, b, a_scale, b_scale, m, n, k,
                                     scale_major, i, j);
            uint16_t bits;
            round_one(r, out_dtype, &bits);
            if (ref)
                ref[i * n + j] = r;
            if (out)
                out[i * n + j] = bits;
        }
    }
    return 0;
}

int oracle_gemm_nt_groupwise_at(const uint8_t* a, const uint8_t* b,
                                const float* a_scale, const float* b_scale,
                                int64_t m, int64_t n, int64_t k, int scale_major,
                                int out_dtype, const int64_t* rows,
                                const int64_t* cols, int64_t count,
                                double* ref, uint16_t* out)
{
    if (check_dense_shape(m, n, k, scale_major, out_dtype) || count < 0)
        return -1;
    for (int64_t s = 0; s < count; ++s)
        if (rows[s] < 0 || rows[s] >= m || cols[s] < 0 || cols[s] >= n)
            return -1;
    double dec[256];
    oracle_e4m3_table(dec);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t s = 0; s < count; ++s) {
        double r = dense_element(dec, a, b, a_scale, b_scale, m, n, k,
                                 scale_major, rows[s], cols[s]);
        uint16_t bits;
        round_one(r, out_dtype, &bits);
        if (ref)
            ref[s] = r;
        if (out)
            out[s] = bits;
    }
    return 0;
}

/* The page requires each expert's rows to sit in a contiguous region aligned
 * to 128 rows, with -1 marking padding.  So every 128-row block holds rows of
 * at most one expert; ids outside [-1, G) or two experts in one block are a
 * precondition violation. */
static int check_m_indices(const int32_t* m_indices, int64_t m,
                           int64_t num_groups)
{
    for (int64_t i0 = 0; i0 < m; i0 += 128) {
        int32_t expert = -1;
        for (int64_t i = i0; i < m && i < i0 + 128; ++i) {
            int32_t e = m_indices[i];
            if (e < -1 || e >= num_groups)
                return -1;
            if (e == -1)
                continue;
            if (expert != -1 && e != expert)
                return -1;
            expert = e;
        }
    }
    return 0;
}

/* Grouped element: row i of a against row j of expert e's weights. */
static double grouped_element(const double* dec, const uint8_t* a,
                              const uint8_t* b, const float* a_scale,
                              const float* b_scale, int64_t n, int64_t k,
                              int32_t e, int64_t i, int64_t j)
{
    int64_t kblocks = k / KBLOCK, nblocks = n / NBLOCK;
    const uint8_t* be = b + (int64_t)e * n * k;
    const float* sbe = b_scale + (int64_t)e * nblocks * kblocks;
    return element(dec, a + i * k, be + j * k, a_scale + i * kblocks, 1,
                   sbe + (j / NBLOCK) * kblocks, 1, kblocks);
}

int oracle_group_gemm_contiguous(const uint8_t* a, const uint8_t* b,
                                 const float* a_scale, const float* b_scale,
                                 const int32_t* m_indices, int64_t m, int64_t n,
                                 int64_t k, int64_t num_groups, double* ref,
                                 uint16_t* out, uint8_t* written)
{
    if (check_dense_shape(m, n, k, ORACLE_SCALE_K_MAJOR, ORACLE_OUT_BF16) ||
        num_groups <= 0)
        return -1;
    if (check_m_indices(m_indices, m, num_groups))
        return -2;
    double dec[256];
    oracle_e4m3_table(dec);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i) {
        int32_t e = m_indices[i];
        if (written)
            for (int64_t j = 0; j < n; ++j)
                written[i * n + j] = (uint8_t)(e != -1);
        if (e == -1)
            continue;
        for (int64_t j = 0; j < n; ++j) {
            double r = grouped_element(dec, a, b, a_scale, b_scale, n, k, e,
                                       i, j);
            uint16_t bits;
            round_one(r, ORACLE_OUT_BF16, &bits);
            if (ref)
                ref[i * n + j] = r;
            if (out)
                out[i * n + j] = bits;
        }
    }
    return 0;
}

int oracle_group_gemm_contiguous_at(const uint8_t* a, const uint8_t* b,
                                    const float* a_scale, const float* b_scale,
                                    const int32_t* m_indices, int64_t m,
                                    int64_t n, int64_t k, int64_t num_groups,
                                    const int64_t* rows, const int64_t* cols,
                                    int64_t count, double* ref, uint16_t* out,
                                    uint8_t* written)
{
    if (check_dense_shape(m, n, k, ORACLE_SCALE_K_MAJOR, ORACLE_OUT_BF16) ||
        num_groups <= 0 || count < 0)
        return -1;
    if (check_m_indices(m_indices, m, num_groups))
        return -2;
    for (int64_t s = 0; s < count; ++s)
        if (rows[s] < 0 || rows[s] >= m || cols[s] < 0 || cols[s] >= n)
            return -1;
    double dec[256];
    oracle_e4m3_table(dec);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t s = 0; s < count; ++s) {
        int32_t e = m_indices[rows[s]];
        if (written)
            written[s] = (uint8_t)(e != -1);
        if (e == -1)
            continue;
        double r = grouped_element(dec, a, b, a_scale, b_scale, n, k, e,
                                   rows[s], cols[s]);
        uint16_t bits;
        round_one(r, ORACLE_OUT_BF16, &bits);
        if (ref)
            ref[s] = r;
        if (out)
            out[s] = bits;
    }
    return 0;
}

/* Valid rows of group g: masked_m[g] clamped to [0, max_m]. */
static int64_t valid_rows(const int32_t* masked_m, int64_t g, int64_t max_m)
{
    int64_t v = masked_m[g];
    if (v < 0)
        v = 0;
    if (v > max_m)
        v = max_m;
    return v;
}

static double masked_element(const double* dec, const uint8_t* a,
                             const uint8_t* b, const float* a_scale,
                             const float* b_scale, int64_t max_m, int64_t n,
                             int64_t k, int64_t g, int64_t r, int64_t j)
{
    int64_t kblocks = k / KBLOCK, nblocks = n / NBLOCK;
    int64_t row = g * max_m + r;
    return element(dec, a + row * k, b + (g * n + j) * k,
                   a_scale + row * kblocks, 1,
                   b_scale + (g * nblocks + j / NBLOCK) * kblocks, 1, kblocks);
}

int oracle_batch_gemm_masked(const uint8_t* a, const uint8_t* b,
                             const float* a_scale, const float* b_scale,
                             const int32_t* masked_m, int64_t num_groups,
                             int64_t max_m, int64_t n, int64_t k, double* ref,
                             uint16_t* out, uint8_t* written)
{
    if (check_dense_shape(max_m, n, k, ORACLE_SCALE_K_MAJOR, ORACLE_OUT_BF16) ||
        num_groups < 0)
        return -1;
    double dec[256];
    oracle_e4m3_table(dec);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t g = 0; g < num_groups; ++g) {
        for (int64_t r = 0; r < max_m; ++r) {
            int64_t base = (g * max_m + r) * n;
            int valid = r < valid_rows(masked_m, g, max_m);
            if (written)
                for (int64_t j = 0; j < n; ++j)
                    written[base + j] = (uint8_t)valid;
            if (!valid)
                continue;
            for (int64_t j = 0; j < n; ++j) {
                double x = masked_element(dec, a, b, a_scale, b_scale, max_m,
                                          n, k, g, r, j);
                uint16_t bits;
                round_one(x, ORACLE_OUT_BF16, &bits);
                if (ref)
                    ref[base + j] = x;
                if (out)
                    out[base + j] = bits;
            }
        }
    }
    return 0;
}

int oracle_batch_gemm_masked_at(const uint8_t* a, const uint8_t* b,
                                const float* a_scale, const float* b_scale,
                                const int32_t* masked_m, int64_t num_groups,
                                int64_t max_m, int64_t n, int64_t k,
                                const int64_t* groups, const int64_t* rows,
                                const int64_t* cols, int64_t count, double* ref,
                                uint16_t* out, uint8_t* written)
{
    if (check_dense_shape(max_m, n, k, ORACLE_SCALE_K_MAJOR, ORACLE_OUT_BF16) ||
        num_groups < 0 || count < 0)
        return -1;
    for (int64_t s = 0; s < count; ++s)
        if (groups[s] < 0 || groups[s] >= num_groups || rows[s] < 0 ||
            rows[s] >= max_m || cols[s] < 0 || cols[s] >= n)
            return -1;
    double dec[256];
    oracle_e4m3_table(dec);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t s = 0; s < count; ++s) {
        int valid = rows[s] < valid_rows(masked_m, groups[s], max_m);
        if (written)
            written[s] = (uint8_t)valid;
        if (!valid)
            continue;
        double x = masked_element(dec, a, b, a_scale, b_scale, max_m, n, k,
                                  groups[s], rows[s], cols[s]);
        uint16_t bits;
        round_one(x, ORACLE_OUT_BF16, &bits);
        if (ref)
            ref[s] = x;
        if (out)
            out[s] = bits;
    }
    return 0;
}

/* ------------------------------------------------------------------ E4M3 */

#define E4M3_P 4
#define E4M3_EMIN (-6)
#define E4M3_MAX 448.0

/* Code of a value already on the E4M3 grid with |y| <= 448. */
static uint8_t e4m3_code_of(double y)
{
    uint8_t sign = signbit(y) ? 0x80 : 0;
    double a = fabs(y);
    if (a == 0.0)
        return sign;
    if (a < ldexp(1.0, E4M3_EMIN)) /* subnormal: a = f * 2^-9 */
        return (uint8_t)(sign | (uint8_t)ldexp(a, 9));
    int e2;
    frexp(a, &e2);
    int lead = e2 - 1; /* a = (1 + f/8) * 2^lead */
    uint8_t f = (uint8_t)(ldexp(a, 3 - lead) - 8.0);
    return (uint8_t)(sign | (uint8_t)((lead + 7) << 3) | f);
}

void oracle_e4m3_encode(const double* x, int64_t count, uint8_t* codes)
{
    for (int64_t s = 0; s < count; ++s) {
        if (isnan(x[s])) {
            codes[s] = 0x7F;
            continue;
        }
        /* round on the grid; anything rounding past 448 saturates */
        double y = round_to_format(x[s], E4M3_P, E4M3_EMIN, E4M3_MAX);
        if (fabs(y) > E4M3_MAX)
            y = copysign(E4M3_MAX, x[s]);
        codes[s] = e4m3_code_of(y);
    }
}

/* ------------------------------------------------- fused add RMSNorm + quant */

static double bf16_value(uint16_t bits)
{
    union {
        uint32_t u;
        float f;
    } v;
    v.u = (uint32_t)bits << 16;
    return (double)v.f;
}

/* Row-major 1 x 128 FP8 quantisation of `cols` values: per block of 128,
 * scale = FP32(amax / 448) and code = E4M3(FP32(x / scale)) (an FP64 quotient
 * of two FP32 values rounded to FP32 is the correctly rounded FP32 quotient);
 * an all-zero block gets scale 0 and codes 0. */
static void quant_row_1x128(const double* x, int64_t cols, uint8_t* codes, float* scales)
{
    for (int64_t b = 0; b < cols / KBLOCK; ++b) {
        double amax = 0.0;
        for (int64_t j = b * KBLOCK; j < (b + 1) * KBLOCK; ++j)
            if (fabs(x[j]) > amax)
                amax = fabs(x[j]);
        float scale = (float)(amax / 448.0);
        scales[b] = scale;
        for (int64_t j = b * KBLOCK; j < (b + 1) * KBLOCK; ++j) {
            double q = 0.0;
            if (amax > 0.0)
                q = (double)(float)(x[j] / (double)scale);
            oracle_e4m3_encode(&q, 1, &codes[j]);
        }
    }
}

void oracle_quant_1x128(const double* x, int64_t rows, int64_t cols, uint8_t* codes,
                        float* scales)
{
    if (cols % KBLOCK)
        return;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i)
        quant_row_1x128(x + i * cols, cols, codes + i * cols, scales + i * (cols / KBLOCK));
}

int oracle_fused_add_rmsnorm_fp8_block_quant(const uint16_t* input,
                                             const uint16_t* residual,
                                             const uint16_t* weight, double eps,
                                             int64_t rows, int64_t hidden,
                                             uint16_t* residual_out,
                                             uint16_t* normed_out, uint8_t* out,
                                             float* block_scale)
{
    if (rows < 0 || hidden <= 0 || hidden % KBLOCK)
        return -1;
    const int64_t nblk = hidden / KBLOCK;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < rows; ++i) {
        const uint16_t* in = input + i * hidden;
        const uint16_t* res = residual + i * hidden;
        uint16_t* rout = residual_out + i * hidden;
        uint16_t* nout = normed_out + i * hidden;
        /* the sum of two BF16 values is exact in FP64; one rounding to BF16 */
        double ss = 0.0;
        for (int64_t j = 0; j < hidden; ++j) {
            double x = round_one(bf16_value(in[j]) + bf16_value(res[j]),
                                 ORACLE_OUT_BF16, &rout[j]);
            ss += x * x;
        }
        double r = 1.0 / sqrt(ss / (double)hidden + eps);
        double* y = (double*)malloc(sizeof(double) * (size_t)hidden);
        for (int64_t j = 0; j < hidden; ++j) {
            double x = bf16_value(rout[j]);
            y[j] = round_one(x * r * bf16_value(weight[j]), ORACLE_OUT_BF16, &nout[j]);
        }
        quant_row_1x128(y, hidden, out + i * hidden, block_scale + i * nblk);
        free(y);
    }
    return 0;
}

/* ------------------------------------------- DeepSeek FP8 block-scale MoE */

/* One GEMV row of the groupwise definition: sum over K blocks of the exact
 * block sum times (x_scale[kb] * w_scale[kb]); w is one row of k codes. */
static double block_scaled_dot(const double* dec, const uint8_t* xq, const float* xs,
                               const uint8_t* w, const float* ws, int64_t k)
{
    double r = 0.0;
    for (int64_t kb = 0; kb < k / KBLOCK; ++kb) {
        double p = 0.0;
        for (int64_t t = kb * KBLOCK; t < (kb + 1) * KBLOCK; ++t)
            p += dec[xq[t]] * dec[w[t]];
        r += p * ((double)xs[kb] * (double)ws[kb]);
    }
    return r;
}

/* SwiGLU of one routed row h (BF16 encodings: gate h[0, inter), up
 * h[inter, 2 inter)), act = silu(gate) * up with silu(g) = g / (1 + e^-g) in
 * FP64, then its 1 x 128 quantisation. */
static void swiglu_quant_row(const uint16_t* h, int64_t inter, double* act, uint8_t* codes,
                             float* scales)
{
    for (int64_t j = 0; j < inter; ++j) {
        const double g = bf16_value(h[j]);
        act[j] = g / (1.0 + exp(-g)) * bf16_value(h[inter + j]);
    }
    quant_row_1x128(act, inter, codes, scales);
}

int oracle_moe_swiglu_quant(const uint16_t* h, int64_t rows, int64_t inter, uint8_t* codes,
                            float* scales)
{
    if (rows < 0 || inter <= 0 || inter % KBLOCK)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double* act = (double*)malloc(sizeof(double) * (size_t)inter);
        swiglu_quant_row(h + r * 2 * inter, inter, act, codes + r * inter,
                         scales + r * (inter / KBLOCK));
        free(act);
    }
    return 0;
}

int oracle_moe_combine(const uint16_t* y, const int32_t* row_of, int64_t tokens, int64_t top_k,
                       int64_t hidden, uint16_t* out)
{
    if (tokens < 0 || top_k <= 0 || hidden <= 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < tokens; ++t)
        for (int64_t j = 0; j < hidden; ++j) {
            /* a sum of BF16 values is exact in FP64 here; one rounding */
            double acc = 0.0;
            for (int64_t s = 0; s < top_k; ++s) {
                const int32_t r = row_of[t * top_k + s];
                if (r >= 0)
                    acc += bf16_value(y[(int64_t)r * hidden + j]);
            }
            round_one(acc, ORACLE_OUT_BF16, &out[t * hidden + j]);
        }
    return 0;
}

int oracle_moe_deepseek_fp8_block_scale(const uint16_t* input, const int32_t* token_selected,
                                        const uint8_t* w1, const uint8_t* w2,
                                        const float* s1, const float* s2, int64_t num_tokens,
                                        int64_t num_experts, int64_t top_k, int64_t hidden,
                                        int64_t inter, uint16_t* out)
{
    if (num_tokens < 0 || num_experts <= 0 || top_k <= 0 || hidden <= 0 || inter <= 0 ||
        hidden % KBLOCK || inter % KBLOCK)
        return -1;
    for (int64_t p = 0; p < num_tokens * top_k; ++p)
        if (token_selected[p] < -1 || token_selected[p] >= num_experts)
            return -2;
    const int64_t hb = hidden / KBLOCK, ib = inter / KBLOCK;
    double dec[256];
    oracle_e4m3_table(dec);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < num_tokens; ++t) {
        double* x = (double*)malloc(sizeof(double) * (size_t)hidden);
        uint8_t* xq = (uint8_t*)malloc((size_t)hidden);
        float* xs = (float*)malloc(sizeof(float) * (size_t)hb);
        uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(2 * inter));
        double* act = (double*)malloc(sizeof(double) * (size_t)inter);
        uint8_t* aq = (uint8_t*)malloc((size_t)inter);
        float* as = (float*)malloc(sizeof(float) * (size_t)ib);
        double* acc = (double*)calloc((size_t)hidden, sizeof(double));
        /* the token's activations, quantised 1 x 128 */
        for (int64_t j = 0; j < hidden; ++j)
            x[j] = bf16_value(input[t * hidden + j]);
        quant_row_1x128(x, hidden, xq, xs);
        for (int64_t s = 0; s < top_k; ++s) {
            const int64_t e = token_selected[t * top_k + s];
            if (e < 0)
                continue;
            /* fc1 -> BF16; rows [0, inter) of the expert's fc1 are the gate,
             * rows [inter, 2 inter) the up projection */
            for (int64_t j = 0; j < 2 * inter; ++j) {
                const uint8_t* wr = w1 + (e * 2 * inter + j) * hidden;
                const float* sr = s1 + (e * (2 * inter / KBLOCK) + j / KBLOCK) * hb;
                round_one(block_scaled_dot(dec, xq, xs, wr, sr, hidden), ORACLE_OUT_BF16, &h[j]);
            }
            /* SwiGLU and its 1 x 128 quantisation */
            swiglu_quant_row(h, inter, act, aq, as);
            /* fc2 -> BF16, summed over the token's experts */
            for (int64_t j = 0; j < hidden; ++j) {
                const uint8_t* wr = w2 + (e * hidden + j) * inter;
                const float* sr = s2 + (e * hb + j / KBLOCK) * ib;
                acc[j] += round_one(block_scaled_dot(dec, aq, as, wr, sr, inter),
                                    ORACLE_OUT_BF16, NULL);
            }
        }
        for (int64_t j = 0; j < hidden; ++j)
            round_one(acc[j], ORACLE_OUT_BF16, &out[t * hidden + j]);
        free(x); free(xq); free(xs); free(h); free(act); free(aq); free(as); free(acc);
    }
    return 0;
}

/* ---------------------------------------------------------------- bmm_fp8 */

/* E5M2 (float8_e5m2): sign s, exponent field e (bias 15), mantissa field f.
 * e == 0 is subnormal: f * 2^-2 * 2^(1-15); e == 31 is infinity (f == 0) or
 * NaN; otherwise (1 + f/4) * 2^(e-15). */
void oracle_e5m2_table(double out[256])
{
    for (int c = 0; c < 256; ++c) {
        int s = (c >> 7) & 1;
        int e = (c >> 2) & 31;
        int f = c & 3;
        double v;
        if (e == 31)
            v = f == 0 ? INFINITY : NAN;
        else if (e == 0)
            v = ldexp((double)f, -16);
        else
            v = ldexp((double)(4 + f), e - 17);
        out[c] = s ? -v : v;
    }
}

int oracle_bmm_fp8(const uint8_t* a, const uint8_t* b, int a_fmt, int b_fmt,
                   const float* a_scale, int a_channelwise, const float* b_scale,
                   int b_channelwise, int64_t batch, int64_t m, int64_t n, int64_t k,
                   int out_dtype, double* ref, uint16_t* out)
{
    if (batch < 0 || m < 0 || n < 0 || k < 0 || (a_fmt != ORACLE_FP8_E4M3 &&
        a_fmt != ORACLE_FP8_E5M2) || (b_fmt != ORACLE_FP8_E4M3 && b_fmt != ORACLE_FP8_E5M2))
        return -1;
    double deca[256], decb[256];
    if (a_fmt == ORACLE_FP8_E4M3)
        oracle_e4m3_table(deca);
    else
        oracle_e5m2_table(deca);
    if (b_fmt == ORACLE_FP8_E4M3)
        oracle_e4m3_table(decb);
    else
        oracle_e5m2_table(decb);
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (int64_t bb = 0; bb < batch; ++bb)
        for (int64_t i = 0; i < m; ++i) {
            const uint8_t* arow = a + (bb * m + i) * k;
            const double sa = a_channelwise ? (double)a_scale[bb * m + i] : (double)a_scale[0];
            for (int64_t j = 0; j < n; ++j) {
                /* column j of B (batch bb) is b[bb][t][j], t = 0 .. k-1 */
                double acc = 0.0;
                for (int64_t t = 0; t < k; ++t)
                    acc += deca[arow[t]] * decb[b[(bb * k + t) * n + j]];
                const double sb =
                    b_channelwise ? (double)b_scale[bb * n + j] : (double)b_scale[0];
                const double x = acc * (sa * sb);
                const int64_t o = (bb * m + i) * n + j;
                uint16_t bits;
                double y = round_one(x, out_dtype, &bits);
                (void)y;
                if (ref)
                    ref[o] = x;
                if (out)
                    out[o] = bits;
            }
        }
    return 0;
}
