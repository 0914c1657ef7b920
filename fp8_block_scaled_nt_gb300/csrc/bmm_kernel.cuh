// bmm_fp8 of the MATE page "FlashInfer Wrapper APIs", section GEMM, for sm_103a:
//   out[b] = (A[b] @ B[b]) * a_scale * b_scale
// with A (batch, m, k) and B (batch, k, n) row-major FP8 (each E4M3 or E5M2)
// and FP32 scales that are one tensorwise value or channelwise — per row of A,
// per column of B.  Such scales factor out of the sum over k, so unlike the
// groupwise GEMM (gemm_kernel.cuh) nothing has to be promoted per K block: the
// tensor cores accumulate the whole of K in TMEM and the scales are applied
// once per output, in the epilogue.
//
// Persistent, one CTA per SM, 384 threads, 128 x 256 output tiles:
//   warp 0      TMA producer: per 128-K block an A tile (128 rows x 128 k,
//               K-major) and B as two 128-column halves of 128 k-rows of the
//               tile's batch (the operand stays N-major, as B is stored), into
//               a 4-slot ring.  n and k need only be multiples of 16: the last
//               K block's k past k, and columns past n, read as zero.
//   warp 1      MMA issuer (one thread): per tile KB x 4 tcgen05.mma (K = 32)
//               accumulating into TMEM buffer (tile index mod 2) of 256
//               columns, B read as an MN-major operand; one commit per tile.
//               One thread walks the ring of slots in order: an mbarrier parity
//               wait only tells consecutive phases apart, so a second issuer
//               starting a tile KB blocks ahead would take an old phase of a
//               slot for the new one.  With no promotion between K blocks the
//               issuer has nothing else to wait for, so one keeps the pipe fed.
//   warps 4-11  epilogue: read the tile's FP32 sums from TMEM once, multiply by
//               a_scale(row) * b_scale(column), round to BF16/FP16 through the
//               shared-memory staging slice (store_tile_rows: rows past m and
//               columns past n are not written), release the buffer.
//   warps 2-3   idle (they complete warpgroup 0 for the register split).
// The two buffers let the next tile's MMAs run while a tile's epilogue runs.
// Every pipeline wait is bounded as in gemm_kernel.cuh.
#pragma once

#include "gemm_kernel.cuh"

namespace fp8g {

constexpr int BMM_A_BYTES = BLOCK_M * BLOCK_K;         // 16 KB
constexpr int BMM_B_HALF_BYTES = BLOCK_K * 128;        // 128 k-rows x 128 columns: 16 KB
constexpr int BMM_B_BYTES = 2 * BMM_B_HALF_BYTES;      // the tile's 256 columns

// One CTA per 128 x 256 tile, or a CTA pair per 256 x 256 tile (cta_group::2:
// each CTA loads its own 128 rows of A and one 128-column half of B, so each
// SM moves a third fewer operand bytes per MMA).
template <bool PAIR>
struct BmmCfg {
    // ring slots: a pair's slots are a third smaller; six measured 4% faster than four
    static constexpr int STAGES = PAIR ? 6 : 4;
    static constexpr int TILE_M = PAIR ? 2 * BLOCK_M : BLOCK_M;
    static constexpr int B_BYTES = PAIR ? BMM_B_HALF_BYTES : BMM_B_BYTES;  // per CTA
    static constexpr int STAGE_BYTES = BMM_A_BYTES + B_BYTES;
    static constexpr size_t SMEM_BYTES =
        1024 + size_t(STAGES) * STAGE_BYTES + 2 * OUT_STAGE_BYTES + BAR_BYTES;
    static_assert(SMEM_BYTES <= 232448, "shared memory of the bmm kernel");
};
constexpr size_t BMM_SMEM_BYTES = BmmCfg<false>::SMEM_BYTES;

// Instruction descriptor of kind::f8f6f4: FP32 D; A (format a_fmt, K-major);
// B (format b_fmt, MN-major); M = m (128, or 256 on a pair), N = 256.
// Formats: 0 = E4M3, 1 = E5M2.
__host__ __device__ constexpr uint32_t idesc_bmm(uint32_t a_fmt, uint32_t b_fmt,
                                                 uint32_t m = 128) {
    return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | (0u << 15) | (1u << 16) |
           ((256u >> 3) << 17) | ((m >> 4) << 24);
}

// Shared-memory descriptor of an MN-major operand with 128-byte swizzle: atoms
// of 128 bytes along MN by 8 rows along K (1024 bytes); `lbo` is the distance
// between atoms along MN, `sbo` between 8-row groups along K.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t lbo,
                                                       uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>(lbo >> 4) << 16) | (static_cast<uint64_t>(sbo >> 4) << 32) |
           (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

struct BmmTile {
    int bb;     // batch
    int rin0;   // first row of this CTA's 128 within the batch
    int row0;   // the same row in the (batch * m) x k view of A (and of out)
    int n0;     // first column
};

// Tile t: batch-major, then bands of band_m m-blocks (of TILE_M rows) with the
// m-block fastest.  `rank`: this CTA's half of a pair's 256 rows.
template <bool PAIR>
__device__ __forceinline__ bool bmm_tile(const Params& p, int t, int rank, BmmTile& tile) {
    if (t >= p.num_tiles) return false;
    const int per_batch = p.m_blocks * p.n_tiles;
    const int bb = t / per_batch;
    const int r = t - bb * per_batch;
    const int per_band = p.band_m * p.n_tiles;
    const int band = r / per_band;
    const int rem = r - band * per_band;
    const int in_band = min(p.band_m, p.m_blocks - band * p.band_m);
    const int nb = rem / in_band;
    const int mb = band * p.band_m + rem % in_band;
    tile.bb = bb;
    tile.rin0 = mb * BmmCfg<PAIR>::TILE_M + rank * BLOCK_M;
    tile.row0 = bb * p.rows + tile.rin0;
    tile.n0 = nb * BLOCK_N;
    return true;
}

template <bool PAIR>
__device__ __forceinline__ void bmm_producer(const CUtensorMap* map_a, const CUtensorMap* map_b,
                                             const Params& p, int rank, uint8_t* sA, uint8_t* sB,
                                             uint64_t* full, uint64_t* empty, const Ctl& ctl) {
    using C = BmmCfg<PAIR>;
    const int lane = threadIdx.x & 31;
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    for (int t = tile_first<PAIR>(); ok; t += tile_stride<PAIR>()) {
        BmmTile tile;
        if (!bmm_tile<PAIR>(p, t, rank, tile)) break;
        if (lane == 0) {
            for (int kb = 0; kb < p.kblocks; ++kb) {
                if (!wait_phase(empty + stage, phase ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full + stage, C::STAGE_BYTES);
                tma_load_2d(sA + stage * BMM_A_BYTES, map_a, full + stage, kb * BLOCK_K,
                            tile.row0);
                uint8_t* b = sB + stage * C::B_BYTES;
                if constexpr (PAIR) {
                    // this CTA's 128-column half of the pair's 256 columns
                    tma_load_3d(b, map_b, full + stage, tile.n0 + rank * 128, kb * BLOCK_K,
                                tile.bb);
                } else {
                    tma_load_3d(b, map_b, full + stage, tile.n0, kb * BLOCK_K, tile.bb);
                    tma_load_3d(b + BMM_B_HALF_BYTES, map_b, full + stage, tile.n0 + 128,
                                kb * BLOCK_K, tile.bb);
                }
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0)
        for (int s = 0; s < C::STAGES; ++s)
            if ((armed >> s) & 1u) drain_wait(full + s, (armed_parity >> s) & 1u);
    __syncwarp();
}

// Odd CTA of a pair: each time one of its slots has landed, arrive on the even
// CTA's barrier of that slot, whose MMA warp then sees both halves land.
__device__ __forceinline__ void bmm_relay(const Params& p, uint64_t* full, const Ctl& ctl) {
    const int lane = threadIdx.x & 31;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = tile_first<true>(); ok; t += tile_stride<true>()) {
        BmmTile tile;
        if (!bmm_tile<true>(p, t, 1, tile)) break;
        if (lane == 0) {
            for (int kb = 0; kb < p.kblocks; ++kb) {
                if (!wait_phase(full + stage, phase, ctl)) {
                    ok = false;
                    break;
                }
                mbar_arrive_remote(mapa_shared(full + stage, 0));
                if (++stage == BmmCfg<true>::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
    }
}

// Tile tl of this CTA (or pair: issued by the even CTA) goes to TMEM buffer
// tl mod 2, accumulating over the whole of K; slots are taken in order
// j = 0, 1, 2, ...
template <bool PAIR>
__device__ __forceinline__ void bmm_mma(const Params& p, uint8_t* sA, uint8_t* sB, uint64_t* full,
                                        uint64_t* empty, uint64_t* acc_full, uint64_t* acc_empty,
                                        uint64_t* drain, uint32_t tmem_base, const Ctl& ctl) {
    const int lane = threadIdx.x & 31;
    const uint64_t a_desc0 = smem_desc_k_sw128(smem_u32(sA));
    const uint32_t b_base = smem_u32(sB);
    const int KB = p.kblocks;
    uint32_t j = 0, tl = 0;  // K blocks and tiles of this CTA so far
    bool ok = true;
    for (int t = tile_first<PAIR>(); ok; t += tile_stride<PAIR>(), ++tl, j += KB) {
        BmmTile tile;
        if (!bmm_tile<PAIR>(p, t, 0, tile)) break;
        if (lane == 0) {
            const int buf = static_cast<int>(tl & 1u);
            const uint32_t bphase = (tl >> 1) & 1u;
            const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BLOCK_N);
            ok = wait_phase(acc_empty + buf, bphase ^ 1u, ctl);
            for (int kb = 0; ok && kb < KB; ++kb) {
                const uint32_t stage = (j + kb) % BmmCfg<PAIR>::STAGES;
                const uint32_t phase = ((j + kb) / BmmCfg<PAIR>::STAGES) & 1u;
                if (!wait_phase(full + stage, phase, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * BMM_A_BYTES) >> 4);
                const uint32_t bs = b_base + stage * BmmCfg<PAIR>::B_BYTES;
#pragma unroll
                for (int kk = 0; kk < BLOCK_K / UMMA_K; ++kk) {
                    // A: +32 bytes inside its swizzled rows; B: +32 k-rows (4 atoms).
                    // On a pair each CTA's B is one 128-column half (one atom wide).
                    const uint64_t bd = smem_desc_mn_sw128(bs + kk * UMMA_K * 128,
                                                           BMM_B_HALF_BYTES, 1024);
                    const uint64_t adk = ad + static_cast<uint64_t>((kk * UMMA_K) >> 4);
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                    if constexpr (PAIR)
                        umma_f8f6f4_pair(d, adk, bd, p.idesc, acc);
                    else
                        umma_f8f6f4(d, adk, bd, p.idesc, acc);
                }
                if constexpr (PAIR)
                    umma_commit_pair_multicast(empty + stage, 0x3);  // both CTAs' slots
                else
                    umma_commit(empty + stage);
            }
            if (ok) {
                if constexpr (PAIR)
                    umma_commit_pair_multicast(acc_full + buf, 0x3);  // both CTAs' rows
                else
                    umma_commit(acc_full + buf);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
        if constexpr (PAIR)
            umma_commit_pair(drain);
        else
            umma_commit(drain);
        drain_wait(drain, 0);
    }
    __syncwarp();
}

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    return static_cast<uint64_t>(__float_as_uint(lo)) |
           (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

template <typename OutT, bool PAIR>
__device__ __forceinline__ void bmm_epilogue(const Params& p, int rank, uint64_t* acc_full,
                                             uint64_t* acc_empty, uint32_t tmem_base,
                                             uint8_t* sOut, const Ctl& ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int half = (warp - FIRST_PROMO_WARP) >> 2;
    const int r = quarter * 32 + lane;
    OutT* out = static_cast<OutT*>(p.out);
    uint32_t tl = 0;
    for (int t = tile_first<PAIR>();; t += tile_stride<PAIR>(), ++tl) {
        BmmTile tile;
        if (!bmm_tile<PAIR>(p, t, rank, tile)) break;
        const int buf = static_cast<int>(tl & 1u);
        const uint32_t bphase = (tl >> 1) & 1u;
        const int rin = tile.rin0 + r;
        const bool row_ok = rin < p.rows;
        const int col0 = tile.n0 + half * 128;
        const bool col_ok = col0 < p.n;  // uniform over the warpgroup
        const int cols = min(128, p.n - col0);  // columns of this half inside n
        const int64_t out_row = static_cast<int64_t>(tile.bb) * p.rows + rin;
        const float sa = p.a_channelwise
                             ? (row_ok ? __ldg(p.a_scale + static_cast<int64_t>(tile.bb) * p.rows +
                                               rin)
                                       : 0.0f)
                             : __ldg(p.a_scale);
        const float* sb = p.b_channelwise ? p.b_scale + static_cast<int64_t>(tile.bb) * p.n + col0
                                          : p.b_scale;
        const bool ok = warp_wait(acc_full + buf, bphase, ctl);
        uint64_t acc[64];
        if (ok) {
            tc_fence_after_sync();
            if (col_ok) {
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       static_cast<uint32_t>(buf * BLOCK_N + half * 128);
                const float sb1 = p.b_channelwise ? 0.0f : __ldg(sb);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[16];
                    tmem_load_16cols_async(taddr + c * 16, v);
                    tmem_wait_16(v);
                    // n is a multiple of 16: a 16-column chunk is all inside n or
                    // all past it (its channelwise scales do not exist)
                    const bool chunk_in = c * 16 < cols;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float s0 = sb1, s1 = sb1;
                        if (p.b_channelwise) {
                            s0 = chunk_in ? __ldg(sb + c * 16 + 2 * i) : 0.0f;
                            s1 = chunk_in ? __ldg(sb + c * 16 + 2 * i + 1) : 0.0f;
                        }
                        acc[c * 8 + i] = pack_f32x2(__uint_as_float(v[2 * i]) * (sa * s0),
                                                    __uint_as_float(v[2 * i + 1]) * (sa * s1));
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                // a pair's buffers are reused by the even CTA's MMA warp
                if constexpr (PAIR)
                    mbar_arrive_remote(mapa_shared(acc_empty + buf, 0));
                else
                    mbar_arrive(acc_empty + buf);
            }
        }
        if (col_ok)
            store_tile_rows<OutT>(out, p.n, out_row - r, col0, ok && row_ok, acc,
                                  sOut + half * OUT_STAGE_BYTES, 1 + half, 1.0f, cols);
        if (named_barrier_or(1 + half, 128, !ok)) break;
    }
}

template <typename OutT, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bmm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const Params p) {
    using C = BmmCfg<PAIR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + C::STAGES * BMM_A_BYTES;
    uint8_t* sOut = sB + C::STAGES * C::B_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sOut + 2 * OUT_STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* acc_full = empty + C::STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            // the even CTA of a pair also counts the odd CTA's relay
            mbar_init(full + s, (PAIR && rank == 0) ? 2 : 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, PAIR ? 2 * NUM_PROMO_WARPS : NUM_PROMO_WARPS);
        }
        mbar_init(drain, 1);  // the MMA issuer's final commit
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    if constexpr (PAIR)
        cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    const Ctl ctl{abort_flag, PAIR ? mapa_shared(abort_flag, rank ^ 1) : 0u, p.status,
                  p.wait_limit_ns};
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp < FIRST_PROMO_WARP) {
        regs_dec<CONTROL_REGS>();
        if (warp == 0) {
            bmm_producer<PAIR>(&map_a, &map_b, p, rank, sA, sB, full, empty, ctl);
        } else if (warp == 1) {
            if (PAIR && rank == 1)
                bmm_relay(p, full, ctl);
            else
                bmm_mma<PAIR>(p, sA, sB, full, empty, acc_full, acc_empty, drain, tmem_base, ctl);
        }
    } else {
        regs_inc<PROMO_REGS>();
        bmm_epilogue<OutT, PAIR>(p, rank, acc_full, acc_empty, tmem_base, sOut, ctl);
    }

    tc_fence_before_sync();
    if constexpr (PAIR)
        cluster_sync();  // no CTA leaves while the other may still signal it
    else
        __syncthreads();
    if (*reinterpret_cast<volatile int*>(abort_flag)) {
        abort_grace();
        if constexpr (PAIR)
            cluster_sync();
        else
            __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace fp8g
