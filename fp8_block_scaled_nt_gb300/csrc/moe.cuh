// The DeepSeek FP8 block-scale MoE layer ("flashinfer-rs" page, section "API
// Example: Fused MoE FP8 (cudarc)", DeepSeek FP8 block-scale mode) around the
// contiguous grouped GEMM of the MATE page "FlashInfer Wrapper APIs", section
// GEMM (group_deepgemm_fp8_nt_groupwise).  For each token t and each of its
// top_k slots with expert e = token_selected[t, s] (-1: empty slot):
//   h   = BF16(fc1_e(Q(input[t])))      fc1 (E, 2 I, H); rows [0, I) are the
//                                       gate, rows [I, 2 I) the up projection
//   act = silu(h_gate) * h_up           (FP32)
//   y   = BF16(fc2_e(Q(act)))           fc2 (E, H, I)
//   out[t] = BF16(sum over the slots of y)
// with Q the row-major 1 x 128 E4M3 quantisation (scale = amax / 448) and the
// GEMMs groupwise-scaled at (1, 128, 128) with 128 x 128 weight-block scales.
//
// The steps, each a kernel on the caller's stream:
//   moe_route_kernel          expert histogram, 128-row-aligned segment offsets,
//                             slot -> row map and m_indices (-1 = padding)
//   moe_quant_gather_kernel   Q of each token, written to its slots' rows
//   gemm_kernel<grouped>      fc1 into h (M x 2 I, BF16)
//   moe_swiglu_quant_kernel   act and its Q for every routed row
//   gemm_kernel<grouped>      fc2 into y (M x H, BF16)
//   moe_combine_kernel        out[t] = sum of the token's rows of y
// M = round_up(tokens * top_k + 127 * E, 128) rows bound every layout; the
// GEMMs skip blocks that hold only padding.  The order of rows inside an
// expert's segment depends on atomics; no result depends on it (every row is
// computed on its own and the combine sums in slot order).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "fp8g.h"
#include "norm_quant.cuh"
#include "ptx.cuh"

namespace fp8g {

constexpr int MOE_ROUTE_THREADS = 1024;
constexpr int MOE_ROW_THREADS = 128;  // per token / per routed row
constexpr int MOE_MAX_EXPERTS = 4096;
// Loads a thread issues before it uses the first of them: these kernels are
// bound by memory latency, so every thread keeps this many reads in flight.
constexpr int MOE_ROUTE_BATCH = 8;
constexpr int MOE_ROW_BATCH = 4;
constexpr int MOE_COMBINE_SLOTS = 8;  // slots whose rows the combine reads at once

__host__ __device__ inline int64_t moe_rows(int64_t tokens, int64_t top_k, int64_t experts) {
    return (tokens * top_k + 127 * experts + 127) / 128 * 128;
}

// One CTA.  Shared memory: counts, offsets and cursors of the experts.  The
// slots are read twice (to count, then to place); m_indices is written from
// the segments' offsets and counts in coalesced runs, not slot by slot.
__global__ void __launch_bounds__(MOE_ROUTE_THREADS)
    moe_route_kernel(const int32_t* __restrict__ token_selected, int pairs, int experts,
                     int m_rows, int32_t* __restrict__ m_indices, int32_t* __restrict__ row_of,
                     unsigned int* status) {
    extern __shared__ int route_smem[];
    __shared__ int warp_total[MOE_ROUTE_THREADS / 32];
    int* count = route_smem;
    int* offset = route_smem + experts;
    int* cursor = route_smem + 2 * experts;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    grid_dependency_wait();
    grid_launch_dependents();
    for (int e = threadIdx.x; e < experts; e += blockDim.x) count[e] = cursor[e] = 0;
    __syncthreads();
    for (int p0 = threadIdx.x; p0 < pairs; p0 += blockDim.x * MOE_ROUTE_BATCH) {
        int e[MOE_ROUTE_BATCH];
#pragma unroll
        for (int u = 0; u < MOE_ROUTE_BATCH; ++u) {
            const int p = p0 + u * blockDim.x;
            e[u] = p < pairs ? __ldg(token_selected + p) : -1;
        }
#pragma unroll
        for (int u = 0; u < MOE_ROUTE_BATCH; ++u) {
            if (e[u] >= 0 && e[u] < experts)
                atomicAdd(&count[e[u]], 1);
            else if (e[u] != -1)
                atomicOr(status, FP8G_DEVICE_BAD_M_INDICES);
        }
    }
    __syncthreads();
    // offsets: exclusive scan of the counts rounded up to 128, the experts split
    // evenly over the threads (every thread runs the shuffles)
    const int per = (experts + blockDim.x - 1) / blockDim.x;
    const int e0 = min(experts, static_cast<int>(threadIdx.x) * per);
    const int e1 = min(experts, e0 + per);
    int mine = 0;
    for (int e = e0; e < e1; ++e) mine += (count[e] + 127) / 128 * 128;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_total[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = static_cast<int>(blockDim.x) / 32;
        int t = lane < nw ? warp_total[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += v;
        }
        if (lane < nw) warp_total[lane] = t;  // inclusive over the warps
    }
    __syncthreads();
    int acc = incl - mine + (warp > 0 ? warp_total[warp - 1] : 0);
    for (int e = e0; e < e1; ++e) {
        offset[e] = acc;
        acc += (count[e] + 127) / 128 * 128;
    }
    __syncthreads();
    for (int p0 = threadIdx.x; p0 < pairs; p0 += blockDim.x * MOE_ROUTE_BATCH) {
        int e[MOE_ROUTE_BATCH];
#pragma unroll
        for (int u = 0; u < MOE_ROUTE_BATCH; ++u) {
            const int p = p0 + u * blockDim.x;
            e[u] = p < pairs ? __ldg(token_selected + p) : -1;
        }
#pragma unroll
        for (int u = 0; u < MOE_ROUTE_BATCH; ++u) {
            const int p = p0 + u * blockDim.x;
            if (p >= pairs) break;
            int row = -1;
            if (e[u] >= 0 && e[u] < experts) row = offset[e[u]] + atomicAdd(&cursor[e[u]], 1);
            row_of[p] = row;
        }
    }
    // m_indices segment by segment, one warp per expert: its rows, then -1 up to
    // the next multiple of 128; then -1 past the last segment
    const int nwarps = static_cast<int>(blockDim.x) / 32;
    for (int e = warp; e < experts; e += nwarps) {
        const int start = offset[e], n = count[e], len = (n + 127) / 128 * 128;
        for (int i = lane; i < len; i += 32) m_indices[start + i] = i < n ? e : -1;
    }
    const int total = offset[experts - 1] + (count[experts - 1] + 127) / 128 * 128;
    for (int r = total + static_cast<int>(threadIdx.x); r < m_rows; r += blockDim.x)
        m_indices[r] = -1;
}

// 1 x 128 quantisation of 8 FP32 values held by each of the 16 lanes of a
// half-warp (one 128-column block): codes (8 bytes per lane) and the scale.
__device__ __forceinline__ uint2 quantise_block_8(const float (&v)[8], unsigned half_mask,
                                                  float& scale) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, o));
    const bool zero = amax == 0.0f;
    scale = zero ? 0.0f : __fdiv_rn(amax, 448.0f);
    const BlockDivisor div(scale);
    uint2 codes;
    codes.x = e4m3_pair(v[0], v[1], div, zero) | (e4m3_pair(v[2], v[3], div, zero) << 16);
    codes.y = e4m3_pair(v[4], v[5], div, zero) | (e4m3_pair(v[6], v[7], div, zero) << 16);
    return codes;
}

// One CTA per token: Q(input[t]) written to the rows of the token's slots.
__global__ void __launch_bounds__(MOE_ROW_THREADS)
    moe_quant_gather_kernel(const uint16_t* __restrict__ input,
                            const int32_t* __restrict__ row_of, int top_k, int hidden,
                            uint8_t* __restrict__ a, float* __restrict__ a_scale) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int t = blockIdx.x;
    const int nblk = hidden / NQ_BLOCK;
    const int lane = threadIdx.x & 31, hl = threadIdx.x & 15;
    const unsigned half_mask = 0xFFFFu << (lane & 16);
    const uint4* in4 = reinterpret_cast<const uint4*>(input + static_cast<int64_t>(t) * hidden);
    constexpr int STEP = MOE_ROW_THREADS / 16;  // blocks per pass of the CTA
    for (int blk0 = threadIdx.x >> 4; blk0 < nblk; blk0 += STEP * MOE_ROW_BATCH) {
        uint4 x[MOE_ROW_BATCH];
#pragma unroll
        for (int u = 0; u < MOE_ROW_BATCH; ++u) {
            const int blk = blk0 + u * STEP;
            if (blk < nblk) x[u] = ld_once_ro_v4(in4 + blk * (NQ_BLOCK / 8) + hl);
        }
#pragma unroll
        for (int u = 0; u < MOE_ROW_BATCH; ++u) {
            const int blk = blk0 + u * STEP;  // uniform over the half-warp
            if (blk >= nblk) break;
            const int v = blk * (NQ_BLOCK / 8) + hl;
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&x[u]);
            float f[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) f[2 * i] = bf16_lo(xw[i]), f[2 * i + 1] = bf16_hi(xw[i]);
            float scale;
            const uint2 codes = quantise_block_8(f, half_mask, scale);
            for (int s = 0; s < top_k; ++s) {
                const int r = __ldg(row_of + static_cast<int64_t>(t) * top_k + s);
                if (r < 0) continue;
                reinterpret_cast<uint2*>(a + static_cast<int64_t>(r) * hidden)[v] = codes;
                if (hl == 0) a_scale[static_cast<int64_t>(r) * nblk + blk] = scale;
            }
        }
    }
}

// One CTA per row of the layout; padding rows are skipped.
__global__ void __launch_bounds__(MOE_ROW_THREADS)
    moe_swiglu_quant_kernel(const uint16_t* __restrict__ h, const int32_t* __restrict__ m_indices,
                            int inter, uint8_t* __restrict__ a, float* __restrict__ a_scale) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int row = blockIdx.x;
    if (__ldg(m_indices + row) < 0) return;
    const int nblk = inter / NQ_BLOCK;
    const int lane = threadIdx.x & 31, hl = threadIdx.x & 15;
    const unsigned half_mask = 0xFFFFu << (lane & 16);
    const uint4* g4 = reinterpret_cast<const uint4*>(h + static_cast<int64_t>(row) * 2 * inter);
    const uint4* u4 = g4 + inter / 8;
    for (int blk = threadIdx.x >> 4; blk < nblk; blk += MOE_ROW_THREADS / 16) {
        const int v = blk * (NQ_BLOCK / 8) + hl;
        const uint4 gv = ld_once_v4(g4 + v);
        const uint4 uv = ld_once_v4(u4 + v);
        const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv);
        const uint32_t* uw = reinterpret_cast<const uint32_t*>(&uv);
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // silu(g) = g / (1 + e^-g) with the fast exponential and divide
            // (a few units in the last place; the kernel is bound by these
            // instructions, the IEEE forms took twice as many)
            const float g0 = bf16_lo(gw[i]), g1 = bf16_hi(gw[i]);
            f[2 * i] = __fdividef(g0, 1.0f + __expf(-g0)) * bf16_lo(uw[i]);
            f[2 * i + 1] = __fdividef(g1, 1.0f + __expf(-g1)) * bf16_hi(uw[i]);
        }
        float scale;
        const uint2 codes = quantise_block_8(f, half_mask, scale);
        reinterpret_cast<uint2*>(a + static_cast<int64_t>(row) * inter)[v] = codes;
        if (hl == 0) a_scale[static_cast<int64_t>(row) * nblk + blk] = scale;
    }
}

// One CTA per token: out[t] = BF16(sum over the token's slots of y[row]),
// summed in FP32 in slot order; a token without a valid slot gets zeros.
__global__ void __launch_bounds__(MOE_ROW_THREADS)
    moe_combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ row_of,
                       int top_k, int hidden, uint16_t* __restrict__ out) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int t = blockIdx.x;
    const int nvec = hidden / 8;
    const int32_t* rows = row_of + static_cast<int64_t>(t) * top_k;
    for (int v = threadIdx.x; v < nvec; v += MOE_ROW_THREADS) {
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        // slots in groups of MOE_COMBINE_SLOTS: all of a group's rows are read
        // before the first is added (the sum stays in slot order)
        for (int s0 = 0; s0 < top_k; s0 += MOE_COMBINE_SLOTS) {
            uint4 yv[MOE_COMBINE_SLOTS];
            bool live[MOE_COMBINE_SLOTS];
#pragma unroll
            for (int j = 0; j < MOE_COMBINE_SLOTS; ++j) {
                const int r = s0 + j < top_k ? __ldg(rows + s0 + j) : -1;
                live[j] = r >= 0;
                if (live[j])
                    yv[j] = ld_once_v4(reinterpret_cast<const uint4*>(
                                           y + static_cast<int64_t>(r) * hidden) + v);
            }
#pragma unroll
            for (int j = 0; j < MOE_COMBINE_SLOTS; ++j) {
                if (!live[j]) continue;
                const uint32_t* yw = reinterpret_cast<const uint32_t*>(&yv[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] += bf16_lo(yw[i]);
                    acc[2 * i + 1] += bf16_hi(yw[i]);
                }
            }
        }
        uint4 o;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) ow[i] = bf16_pack(acc[2 * i], acc[2 * i + 1]);
        reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * hidden)[v] = o;
    }
}

}  // namespace fp8g
