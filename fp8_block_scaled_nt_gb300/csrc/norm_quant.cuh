// Fused add + RMSNorm + row-major 1 x 128 FP8 (E4M3) quantisation for sm_103a:
// fused_add_rmsnorm_fp8_block_quant of the MATE page "FlashInfer Wrapper
// APIs", section Norm.  It produces the GEMM's FP8 activations and their
// K-major (1, 128) scales in one pass over HBM.
//
// Per row of `hidden` BF16 values:
//   x_j      = BF16(input_j + residual_j)           -> residual (in place)
//   r        = 1 / sqrt(mean_j x_j^2 + eps)         (FP32)
//   y_j      = BF16(x_j * r * weight_j)             -> normed_out
//   per 128-column block: amax = max |y_j|, scale = amax / 448 (FP32, IEEE
//   division) -> block_scale; code_j = E4M3(y_j / scale) with round to
//   nearest even and saturation at +-448 -> out.  An all-zero block gets scale
//   0 and codes 0.
// The kernel is bound by HBM bandwidth: per element it reads 4 bytes (input,
// residual) and writes 5 (residual, normed_out, out), plus the weight row,
// which stays in L2, and 4 bytes of scale per 128 elements.
//
// Rows of up to 8192 elements run on a persistent kernel that pulls each row
// with two bulk copies into a two-slot shared-memory ring (below); longer rows
// run one CTA per row, where pass 1 streams input and residual with 16-byte loads,
// writes the new residual, keeps x in shared memory and reduces the sum of
// squares; pass 2 gives each 128-column block to a half-warp (8 values per
// lane), which normalises, finds the block's amax with four shuffles and
// writes normed_out, the codes and the scale.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "fp8g.h"
#include "ptx.cuh"

namespace fp8g {

constexpr int NQ_THREADS = 256;
constexpr int NQ_BLOCK = 128;  // quantisation block (1 x 128)

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf16_pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 16-byte load of data read once: read-only path for a tensor nobody writes,
// plain load for one this kernel overwrites afterwards.
__device__ __forceinline__ uint4 ld_once_ro_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_once_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// Correctly rounded y / scale for the elements of one 1 x 128 block, by
// Markstein's scheme (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with r
// the correctly rounded reciprocal of scale (once per block), q = y * r is
// within two ulps of y / scale; a correction q += (y - scale q) r, whose
// residual the FMA forms exactly, brings it within one ulp, and by
// Markstein's theorem a second such correction rounds it correctly.  Where a
// step could overflow or underflow (scale outside [2^-100, 2^100]) it falls
// back to the IEEE division.  Quotients too small for the residual to be
// exact lie far below the smallest E4M3 subnormal, where every candidate
// gives the same code.
struct BlockDivisor {
    float b, r;
    bool fast;
    __device__ __forceinline__ explicit BlockDivisor(float scale) : b(scale) {
        fast = scale >= 0x1p-100f && scale <= 0x1p+100f;
        r = fast ? __frcp_rn(scale) : 0.0f;
    }
    __device__ __forceinline__ float operator()(float y) const {
        if (!fast) return __fdiv_rn(y, b);
        float q = y * r;
        q = fmaf(fmaf(-b, q, y), r, q);
        return fmaf(fmaf(-b, q, y), r, q);
    }
};

// Two E4M3 codes of y0 / scale and y1 / scale (low byte first).
__device__ __forceinline__ uint32_t e4m3_pair(float y0, float y1, const BlockDivisor& div,
                                              bool zero) {
    float2 q;
    q.x = zero ? 0.0f : div(y0);
    q.y = zero ? 0.0f : div(y1);
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3));
}

__global__ void __launch_bounds__(NQ_THREADS)
    fused_add_rmsnorm_quant_kernel(uint8_t* __restrict__ out, float* __restrict__ block_scale,
                                   uint16_t* __restrict__ normed_out,
                                   const uint16_t* __restrict__ input,
                                   uint16_t* __restrict__ residual,
                                   const uint16_t* __restrict__ weight, float eps, int rows,
                                   int hidden) {
    extern __shared__ uint4 xs[];  // this row's x, hidden / 8 vectors of 8 BF16
    __shared__ float partial[NQ_THREADS / 32];
    // global memory only after the previous kernel on the stream is done
    grid_dependency_wait();
    grid_launch_dependents();
    const int nvec = hidden / 8;
    const int nblk = hidden / NQ_BLOCK;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t base = static_cast<int64_t>(row) * hidden;
        const uint4* in4 = reinterpret_cast<const uint4*>(input + base);
        uint4* res4 = reinterpret_cast<uint4*>(residual + base);

        // pass 1: x = BF16(input + residual), sum of squares of x
        float ss = 0.0f;
#pragma unroll 4
        for (int v = threadIdx.x; v < nvec; v += NQ_THREADS) {
            const uint4 a = ld_once_ro_v4(in4 + v);
            const uint4 r = ld_once_v4(res4 + v);
            uint4 x;
            uint32_t* xw = reinterpret_cast<uint32_t*>(&x);
            const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
            const uint32_t* rw = reinterpret_cast<const uint32_t*>(&r);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xw[i] = bf16_pack(bf16_lo(aw[i]) + bf16_lo(rw[i]), bf16_hi(aw[i]) + bf16_hi(rw[i]));
                const float lo = bf16_lo(xw[i]), hi = bf16_hi(xw[i]);
                ss = fmaf(lo, lo, ss);
                ss = fmaf(hi, hi, ss);
            }
            res4[v] = x;
            xs[v] = x;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) partial[warp] = ss;
        __syncthreads();  // also publishes xs
        float total = 0.0f;
#pragma unroll
        for (int w = 0; w < NQ_THREADS / 32; ++w) total += partial[w];
        const float rinv = __frsqrt_rn(__fdiv_rn(total, static_cast<float>(hidden)) + eps);

        // pass 2: one 128-column block per half-warp, 8 values per lane
        const int hl = threadIdx.x & 15;
        const unsigned half_mask = 0xFFFFu << (lane & 16);
        const uint4* w4 = reinterpret_cast<const uint4*>(weight);
        uint4* n4 = reinterpret_cast<uint4*>(normed_out + base);
        uint2* o2 = reinterpret_cast<uint2*>(out + base);
        for (int blk = threadIdx.x >> 4; blk < nblk; blk += NQ_THREADS / 16) {
            const int v = blk * (NQ_BLOCK / 8) + hl;
            const uint4 x = xs[v];
            const uint4 wv = __ldg(w4 + v);
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&x);
            const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv);
            uint4 y;
            uint32_t* yw = reinterpret_cast<uint32_t*>(&y);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                yw[i] = bf16_pack(bf16_lo(xw[i]) * rinv * bf16_lo(ww[i]),
                                  bf16_hi(xw[i]) * rinv * bf16_hi(ww[i]));
                amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(yw[i])), fabsf(bf16_hi(yw[i]))));
            }
            n4[v] = y;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, o));
            const bool zero = amax == 0.0f;
            const float scale = zero ? 0.0f : __fdiv_rn(amax, 448.0f);
            const BlockDivisor div(scale);
            uint2 codes;
            codes.x = e4m3_pair(bf16_lo(yw[0]), bf16_hi(yw[0]), div, zero) |
                      (e4m3_pair(bf16_lo(yw[1]), bf16_hi(yw[1]), div, zero) << 16);
            codes.y = e4m3_pair(bf16_lo(yw[2]), bf16_hi(yw[2]), div, zero) |
                      (e4m3_pair(bf16_lo(yw[3]), bf16_hi(yw[3]), div, zero) << 16);
            o2[v] = codes;
            if (hl == 0) block_scale[static_cast<int64_t>(row) * nblk + blk] = scale;
        }
        __syncthreads();  // xs and partial are reused by the next row
    }
}

// The same computation for rows of up to NQR_MAX_HIDDEN elements as a
// persistent kernel: each CTA walks rows blockIdx.x, + gridDim.x, ... and pulls
// every row's input and residual into a ring of NQR_STAGES shared-memory slots
// with two bulk copies (one thread, completion on the slot's mbarrier), the
// next rows' copies in flight while the current row is computed.  The
// arithmetic, and the order of every sum, is that of
// fused_add_rmsnorm_quant_kernel, so the results are bit-identical.
// Two slots and three CTAs per SM (at 7168 columns) beat three slots and two
// CTAs, or four and one (measured: 0.77, 0.63 and 0.40 of the copy bandwidth):
// rows in flight matter more than ring depth.
constexpr int NQR_STAGES = 2;
constexpr int NQR_MAX_HIDDEN = 8192;  // 2 slots x (input + residual) = 64 KB per CTA
constexpr uint64_t NQR_WAIT_LIMIT_NS = 2000000000ull;
constexpr uint64_t NQR_GRACE_NS = 5000000ull;

__global__ void __launch_bounds__(NQ_THREADS)
    fused_add_rmsnorm_quant_ring_kernel(uint8_t* __restrict__ out, float* __restrict__ block_scale,
                                        uint16_t* __restrict__ normed_out,
                                        const uint16_t* __restrict__ input,
                                        uint16_t* __restrict__ residual,
                                        const uint16_t* __restrict__ weight, float eps, int rows,
                                        int hidden, unsigned int* status) {
    // slot s: the row's input (nvec vectors of 8 BF16; pass 1 overwrites it
    // with x), then its residual
    extern __shared__ uint4 ring[];
    __shared__ float partial[NQ_THREADS / 32];
    __shared__ uint64_t full[NQR_STAGES];
    const int nvec = hidden / 8;
    const int nblk = hidden / NQ_BLOCK;
    const uint32_t row_bytes = static_cast<uint32_t>(hidden) * 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NQR_STAGES; ++s) mbar_init(full + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    // global memory only after the previous kernel on the stream is done
    grid_dependency_wait();
    grid_launch_dependents();
    auto fetch = [&](int slot, int row) {
        const int64_t base = static_cast<int64_t>(row) * hidden;
        uint4* dst = ring + static_cast<int64_t>(slot) * 2 * nvec;
        mbar_arrive_expect_tx(full + slot, 2 * row_bytes);
        bulk_load(dst, input + base, row_bytes, full + slot);
        bulk_load(dst + nvec, residual + base, row_bytes, full + slot);
    };
    if (threadIdx.x == 0)
        for (int s = 0; s < NQR_STAGES; ++s)
            if (blockIdx.x + s * gridDim.x < rows) fetch(s, blockIdx.x + s * gridDim.x);
    int it = 0;
    for (int row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
        const int slot = it % NQR_STAGES;
        const uint32_t parity = (it / NQR_STAGES) & 1;
        if (!mbar_try_wait(full + slot, parity)) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(full + slot, parity)) {
                if (global_timer_ns() - t0 > NQR_WAIT_LIMIT_NS) {
                    atomicOr(status, FP8G_DEVICE_TIMEOUT);
                    // copies still in flight land before the shared memory is released
                    const uint64_t t1 = global_timer_ns();
                    while (global_timer_ns() - t1 < NQR_GRACE_NS) {
                    }
                    return;
                }
            }
        }
        const int64_t base = static_cast<int64_t>(row) * hidden;
        uint4* xs = ring + static_cast<int64_t>(slot) * 2 * nvec;
        const uint4* rs = xs + nvec;
        uint4* res4 = reinterpret_cast<uint4*>(residual + base);

        // pass 1: x = BF16(input + residual), sum of squares of x
        float ss = 0.0f;
        for (int v = threadIdx.x; v < nvec; v += NQ_THREADS) {
            const uint4 a = xs[v];
            const uint4 r = rs[v];
            uint4 x;
            uint32_t* xw = reinterpret_cast<uint32_t*>(&x);
            const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
            const uint32_t* rw = reinterpret_cast<const uint32_t*>(&r);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xw[i] = bf16_pack(bf16_lo(aw[i]) + bf16_lo(rw[i]), bf16_hi(aw[i]) + bf16_hi(rw[i]));
                const float lo = bf16_lo(xw[i]), hi = bf16_hi(xw[i]);
                ss = fmaf(lo, lo, ss);
                ss = fmaf(hi, hi, ss);
            }
            res4[v] = x;
            xs[v] = x;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) partial[warp] = ss;
        __syncthreads();  // also publishes xs
        float total = 0.0f;
#pragma unroll
        for (int w = 0; w < NQ_THREADS / 32; ++w) total += partial[w];
        const float rinv = __frsqrt_rn(__fdiv_rn(total, static_cast<float>(hidden)) + eps);

        // pass 2: one 128-column block per half-warp, 8 values per lane
        const int hl = threadIdx.x & 15;
        const unsigned half_mask = 0xFFFFu << (lane & 16);
        const uint4* w4 = reinterpret_cast<const uint4*>(weight);
        uint4* n4 = reinterpret_cast<uint4*>(normed_out + base);
        uint2* o2 = reinterpret_cast<uint2*>(out + base);
        for (int blk = threadIdx.x >> 4; blk < nblk; blk += NQ_THREADS / 16) {
            const int v = blk * (NQ_BLOCK / 8) + hl;
            const uint4 x = xs[v];
            const uint4 wv = __ldg(w4 + v);
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&x);
            const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv);
            uint4 y;
            uint32_t* yw = reinterpret_cast<uint32_t*>(&y);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                yw[i] = bf16_pack(bf16_lo(xw[i]) * rinv * bf16_lo(ww[i]),
                                  bf16_hi(xw[i]) * rinv * bf16_hi(ww[i]));
                amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(yw[i])), fabsf(bf16_hi(yw[i]))));
            }
            n4[v] = y;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, o));
            const bool zero = amax == 0.0f;
            const float scale = zero ? 0.0f : __fdiv_rn(amax, 448.0f);
            const BlockDivisor div(scale);
            uint2 codes;
            codes.x = e4m3_pair(bf16_lo(yw[0]), bf16_hi(yw[0]), div, zero) |
                      (e4m3_pair(bf16_lo(yw[1]), bf16_hi(yw[1]), div, zero) << 16);
            codes.y = e4m3_pair(bf16_lo(yw[2]), bf16_hi(yw[2]), div, zero) |
                      (e4m3_pair(bf16_lo(yw[3]), bf16_hi(yw[3]), div, zero) << 16);
            o2[v] = codes;
            if (hl == 0) block_scale[static_cast<int64_t>(row) * nblk + blk] = scale;
        }
        // the slot (written by this pass, read by the bulk copies) goes back to
        // the async proxy; partial is free for the next row
        fence_proxy_async_shared();
        __syncthreads();
        const int next = row + NQR_STAGES * gridDim.x;
        if (threadIdx.x == 0 && next < rows) fetch(slot, next);
    }
}

}  // namespace fp8g
