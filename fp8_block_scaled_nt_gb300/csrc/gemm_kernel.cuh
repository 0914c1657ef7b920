// Persistent, warp-specialised FP8 (E4M3) groupwise-scaled NT GEMM for sm_103a.
//
// Computes the operation of the MATE page "FlashInfer Wrapper APIs", section
// GEMM (gemm_fp8_nt_groupwise and its grouped/masked MoE forms):
//   out[i][j] = sum_kb P(i,j,kb) * a_scale(i,kb) * b_scale(j/128,kb),
//   P(i,j,kb) = sum over the 128 k of block kb of a[i][k] * b[j][k].
//
// Each CTA owns 128 output rows x 256 columns of a tile at a time.  Per tile
// and per 128-wide K block (one scale block):
//   warp 0      TMA producer: loads this CTA's E4M3 tiles of A and B into a ring
//               of 128-byte-swizzled shared-memory slots.
//   warps 1-2   MMA issuers (even / odd K blocks): 4 x tcgen05.mma (K = 32)
//               write the block's partial sums P into TMEM buffer 0 / 1 (FP32,
//               128 lanes x 256 cols), fresh for every K block.
//   warp 3      storer (dense form): copies each finished tile from its
//               shared-memory staging to global memory with bulk tensor
//               stores; idle in the grouped and masked forms.
//   warps 4-11  promotion: read the partial from TMEM, multiply by
//               a_scale(row,kb) * b_scale(col block,kb) and accumulate in FP32
//               registers (one row per thread, 128 columns per warpgroup);
//               after the last K block round the row to BF16/FP16 (or E4M3)
//               into the staging.  Dense form: hand the staging to the storer
//               and go on with the next tile at once; grouped and masked
//               forms: store the staged rows as whole 128-byte row segments
//               (rows outside the form skipped), 64 columns at a time.
// The 128 x 256 FP32 running sums take half of the register file, so the
// control warpgroup hands registers to the two promotion warpgroups
// (setmaxnreg: 40 + 2 x 232 per thread, exactly the launch's 3 x 168).
// The two TMEM buffers let the tensor cores compute block kb+1 while block kb
// is being promoted.  In the dense form the staging holds a whole tile, so the
// global stores of tile i overlap the promotion of tile i+1 (the storer has a
// whole tile's time to empty it).
//
// Two variants of the pipeline:
//   single CTA  (PAIR = false): a 128 x 256 tile per CTA; the producer loads
//               A 128x128 and B 256x128 (48 KB) per K block into 3 slots (4
//               for the masked form).
//   CTA pair    (PAIR = true, dense form): a cluster of two CTAs computes a
//               256 x 256 tile with tcgen05.mma.cta_group::2 (M = 256).  Each
//               CTA loads its own 128 rows of A and its half (128 rows) of B,
//               32 KB per K block into 4 slots, so every SM moves a third less
//               data through L2 and shared memory per MMA.  The even CTA issues
//               the MMAs and multicasts their completion to both CTAs; the odd
//               CTA's MMA warp relays "my slot has landed" to the even CTA, and
//               its promotion warps release TMEM buffers on the even CTA.
//
// Every wait on a pipeline barrier is bounded: past the limit the waiting warp
// raises an abort flag shared by the CTA and a bit in the device status word,
// all roles leave their loops, in-flight copies and MMAs are drained, TMEM is
// freed and the kernel returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <limits.h>
#include <stdint.h>

#include "fp8g.h"
#include "ptx.cuh"

namespace fp8g {

constexpr int BLOCK_M = 128;  // rows per CTA = TMEM lanes
constexpr int BLOCK_N = 256;  // tile columns = UMMA N
constexpr int BLOCK_K = 128;  // one scale block along k = one 128-byte swizzle row of E4M3
constexpr int UMMA_K = 32;    // K of one kind::f8f6f4 instruction
constexpr int NUM_PROMO_WARPS = 8;
constexpr int FIRST_PROMO_WARP = 4;
constexpr int NUM_THREADS = 128 + 32 * NUM_PROMO_WARPS;  // 3 warpgroups
constexpr uint32_t LAUNCH_REGS = 168;   // per thread at launch (3 warps per SM sub-partition)
constexpr uint32_t CONTROL_REGS = 40;   // warpgroup 0 after setmaxnreg.dec
constexpr uint32_t PROMO_REGS = 232;    // warpgroups 1-2 after setmaxnreg.inc
static_assert(128 * CONTROL_REGS + 256 * PROMO_REGS <= NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch's registers");
constexpr uint32_t TMEM_COLS = 2 * BLOCK_N;  // two FP32 partial buffers
constexpr int BAR_BYTES = 256;  // barriers, TMEM slot, abort flag, storer descriptor
// Output staging of the bmm kernel: each epilogue warpgroup rounds 128 rows x
// 64 columns at a time into 128-byte rows of shared memory before its warps
// store them.
constexpr int OUT_COLS = 64;
constexpr int OUT_STAGE_BYTES = BLOCK_M * OUT_COLS * 2;  // 16 KB per warpgroup
// Output staging of the GEMM kernel: a promotion warpgroup's whole tile share,
// 128 rows x 128 columns, as 128-byte rows (two 64-column slices for BF16/FP16,
// one 128-column slice for E4M3).
constexpr int TILE_STAGE_BYTES = BLOCK_M * 128 * 2;  // 32 KB per warpgroup
constexpr int STAGE_SLICE_BYTES = BLOCK_M * 128;     // one slice of 128-byte rows
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s default: far beyond any legitimate wait
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;
constexpr uint64_t ABORT_GRACE_NS = 5000000ull;  // 5 ms

enum Form { FORM_DENSE = 0, FORM_GROUPED = 1, FORM_MASKED = 2 };

// Grouped form: up to this many 128-row blocks, tiles are ordered expert
// segment by expert segment (a table of segment starts in shared memory);
// beyond it, by bands of band_m blocks.
constexpr int SEG_RASTER_MAX_BLOCKS = 4096;

// Geometry of the pipeline variants.  Ring depths: shared memory left over
// becomes L1, which the per-row scale loads of the promotion warps live on, so
// the rings are as deep as the copies need and no deeper (measured); the
// HBM-bound masked form keeps one more slot in flight.  The dense form hands
// finished tiles to the storer warp through a whole-tile staging (measured:
// +4% on 4096 x 7168 x 2048); the grouped and masked forms keep the shared
// memory for L1 and their rings and store from the promotion warps (the
// storer cost them 1% and 4%).
template <bool PAIR, int FORM>
struct Cfg {
    static constexpr int TILE_M = PAIR ? 2 * BLOCK_M : BLOCK_M;  // rows of a scheduled tile
    static constexpr int B_ROWS = PAIR ? BLOCK_N / 2 : BLOCK_N;  // B rows one CTA loads
    static constexpr int STAGES = PAIR ? 4 : (FORM == FORM_MASKED ? 4 : 3);
    static constexpr bool STORER = FORM == FORM_DENSE;
    static constexpr int OUT_BYTES = STORER ? TILE_STAGE_BYTES : OUT_STAGE_BYTES;  // per half
    static constexpr int A_BYTES = BLOCK_M * BLOCK_K;
    static constexpr int B_BYTES = B_ROWS * BLOCK_K;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // grouped form: the expert-segment table (count, starts, end sentinel)
    static constexpr int SEG_BYTES =
        FORM == FORM_GROUPED ? ((SEG_RASTER_MAX_BLOCKS + 2) * 4 + 15) / 16 * 16 : 0;
    static constexpr size_t SEG_OFFSET = size_t(STAGES) * STAGE_BYTES + 2 * OUT_BYTES;
    static constexpr size_t SMEM_BYTES = 1024 /* alignment slack */ +
                                         size_t(STAGES) * STAGE_BYTES + 2 * OUT_BYTES +
                                         SEG_BYTES + BAR_BYTES;
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
    static constexpr uint32_t IDESC = idesc_e4m3_f32(TILE_M, BLOCK_N);
};

struct Params {
    const float* a_scale;
    const float* b_scale;
    void* out;
    const int32_t* m_indices;  // grouped form
    const int32_t* masked_m;   // masked form
    unsigned int* status;      // device status word
    int rows;                  // dense: m; grouped: M_total; masked: max_m
    int n, k;
    int kblocks, nblocks;  // k/128, n/128 (bmm_fp8: kblocks = ceil(k/128))
    int n_tiles;           // ceil(n / BLOCK_N)
    int m_blocks;          // ceil(rows / TILE_M)
    int num_tiles;         // dense/grouped: m_blocks * n_tiles
    int num_groups;
    int scale_mn_major;  // dense form only
    const float* out_scale;  // dense form with E4M3 output: the output's FP32 scale
    int band_m;          // m-blocks per raster band (dense/grouped)
    int seg_raster;      // grouped: order tiles by expert segment (see Scheduler)
    // bmm_fp8 (bmm_kernel.cuh): rows = m of one batch, k of one batch
    int batch;
    int a_channelwise, b_channelwise;  // scales per row of A / column of B, else one value
    uint32_t idesc;                    // instruction descriptor (operand formats)
    uint64_t wait_limit_ns;            // bound of every pipeline wait (WAIT_LIMIT_NS by default)
};

// One output tile as every role of one CTA sees it.
struct Tile {
    int mb, nb;          // m-block (within the group for the masked form), 256-col block
    int group;           // expert (grouped) or group (masked); 0 for dense
    int row0;            // first of this CTA's 128 rows in the 2-D view of a (and out)
    int b_row0;          // first row of b this CTA loads
    int group_rows;      // masked: valid rows of the group
    int row_expert[4];   // grouped: m_indices of rows 32q + lane, q = 0..3
    bool skip;           // grouped: padding-only block or broken precondition
};

// The kernel's shared memory, 1024-byte aligned (the base every role agrees on).
__device__ __forceinline__ uint8_t* smem_base() {
    extern __shared__ uint8_t smem_raw[];
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
}

// Grouped form: the starts of the runs of 128-row blocks whose first rows carry
// the same m_indices value -- the experts' segments of the contiguous layout
// (and runs of padding-only blocks) -- written by one warp into
// table[1 .. count], with table[0] = count and table[count + 1] = m_blocks.
__device__ __forceinline__ void build_segments(const Params& p, int* table) {
    const int lane = threadIdx.x & 31;
    int count = 0, prev = INT_MIN;
    for (int b0 = 0; b0 < p.m_blocks; b0 += 32) {
        const int b = b0 + lane;
        const int key = b < p.m_blocks ? __ldg(p.m_indices + static_cast<int64_t>(b) * BLOCK_M)
                                       : INT_MIN;
        int left = __shfl_up_sync(0xffffffffu, key, 1);
        if (lane == 0) left = prev;
        const bool start = b < p.m_blocks && (b == 0 || key != left);
        const uint32_t mask = __ballot_sync(0xffffffffu, start);
        if (start) table[1 + count + __popc(mask & ((1u << lane) - 1u))] = b;
        count += __popc(mask);
        prev = __shfl_sync(0xffffffffu, key, 31);
    }
    if (lane == 0) {
        table[0] = count;
        table[1 + count] = p.m_blocks;
    }
}

// Tile ids this CTA (or CTA pair) walks: first, first + stride, ...
template <bool PAIR>
__device__ __forceinline__ int tile_first() {
    if constexpr (PAIR) return static_cast<int>(cluster_id_x());
    return static_cast<int>(blockIdx.x);
}
template <bool PAIR>
__device__ __forceinline__ int tile_stride() {
    if constexpr (PAIR) return static_cast<int>(cluster_count_x());
    return static_cast<int>(gridDim.x);
}

// Maps tile ids to tiles.  All roles walk the same ids through identical
// schedulers, so they agree on every tile.  Called by whole warps (the grouped
// form reduces over the warp).  `rank` is the CTA's rank in its pair (0 for a
// single CTA).
template <int FORM, bool PAIR>
struct Scheduler {
    using C = Cfg<PAIR, FORM>;
    static_assert(!PAIR || FORM != FORM_GROUPED, "CTA pairs serve the dense and masked forms");
    const Params& p;
    const int rank;
    int g = 0;     // masked: group the cursor is in
    int base = 0;  // masked: first tile id of group g
    __device__ Scheduler(const Params& params, int cta_rank) : p(params), rank(cta_rank) {}

    __device__ int masked_rows(int grp, bool flag) const {
        const int v = __ldg(p.masked_m + grp);
        const int c = min(max(v, 0), p.rows);
        if (flag && c != v) atomicOr(p.status, FP8G_DEVICE_MASKED_M_CLAMPED);
        return c;
    }

    // Dense and grouped: raster of bands of `band_m` m-blocks; inside a band the
    // m-block varies fastest, so the CTAs running at one time share A row panels
    // and B column panels in L2.
    __device__ void raster(int t, int& mb, int& nb) const {
        const int per_band = p.band_m * p.n_tiles;
        const int band = t / per_band;
        const int rem = t - band * per_band;
        const int in_band = min(p.band_m, p.m_blocks - band * p.band_m);
        nb = rem / in_band;
        mb = band * p.band_m + rem % in_band;
    }

    // Grouped form: tiles expert segment by expert segment, and within a
    // segment n-block by n-block with the segment's 128-row blocks fastest, so
    // the CTAs running at one time share one expert's weights (which then
    // stream from memory once) and its rows.  The tiles before segment s are
    // n_tiles x its first block.
    __device__ void segment_raster(int t, int& mb, int& nb) const {
        const int* table = reinterpret_cast<const int*>(smem_base() + C::SEG_OFFSET);
        int lo = 0, hi = table[0] - 1;  // the last segment starting at or before t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (table[1 + mid] * p.n_tiles <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int start = table[1 + lo], len = table[2 + lo] - start;
        const int local = t - start * p.n_tiles;
        nb = local / len;
        mb = start + (local - nb * len);
    }

    // False once t is past the last tile.  `flag` lets one thread report
    // precondition violations in the device status word.
    __device__ bool next(int t, Tile& tile, bool flag) {
        tile.skip = false;
        tile.group = 0;
        tile.group_rows = 0;
        if constexpr (FORM == FORM_MASKED) {
            while (g < p.num_groups) {
                const int rows_g = masked_rows(g, flag && blockIdx.x == 0);
                const int mbk = (rows_g + C::TILE_M - 1) / C::TILE_M;
                const int count = mbk * p.n_tiles;
                if (t < base + count) {
                    const int local = t - base;
                    tile.nb = local / mbk;  // m-blocks of one n-block are adjacent ids
                    tile.mb = local - tile.nb * mbk;
                    tile.group = g;
                    tile.group_rows = rows_g;
                    tile.row0 = g * p.rows + tile.mb * C::TILE_M + rank * BLOCK_M;
                    tile.b_row0 = g * p.n + tile.nb * BLOCK_N + rank * C::B_ROWS;
                    return true;
                }
                base += count;
                ++g;
            }
            return false;
        } else {
            if (t >= p.num_tiles) return false;
            if (FORM == FORM_GROUPED && p.seg_raster)
                segment_raster(t, tile.mb, tile.nb);
            else
                raster(t, tile.mb, tile.nb);
            tile.row0 = tile.mb * C::TILE_M + rank * BLOCK_M;
            tile.b_row0 = tile.nb * BLOCK_N + rank * C::B_ROWS;
            if constexpr (FORM == FORM_GROUPED) {
                const int lane = threadIdx.x & 31;
                int lo = INT_MAX, hi = -1, bad = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = tile.row0 + q * 32 + lane;
                    const int e = row < p.rows ? __ldg(p.m_indices + row) : -1;
                    tile.row_expert[q] = e;
                    if (e < -1 || e >= p.num_groups) {
                        bad = 1;
                    } else if (e >= 0) {
                        lo = min(lo, e);
                        hi = max(hi, e);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
                    bad |= __shfl_xor_sync(0xffffffffu, bad, o);
                }
                const bool mixed = hi >= 0 && lo != hi;
                if (flag && (bad || mixed)) atomicOr(p.status, FP8G_DEVICE_BAD_M_INDICES);
                tile.skip = bad || mixed || hi < 0;
                tile.group = hi;
                tile.b_row0 = hi * p.n + tile.nb * BLOCK_N;
            }
            return true;
        }
    }
};

struct Ctl {
    volatile int* abort_flag;  // this CTA's
    uint32_t peer_abort;       // the other CTA's flag in the cluster window (pairs), else 0
    unsigned int* status;
    uint64_t limit_ns;         // give up a wait after this long
};

// Wait for the phase of `bar` with the given parity; false if the CTA aborted
// or this wait exceeded its limit (which aborts this CTA and, in a pair, the
// other CTA too).  The phases are completed by tcgen05 commits, TMA
// transactions or arrivals that follow completed tensor-memory reads, so the
// default (CTA-scope) acquire of try_wait suffices also for pairs.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, const Ctl& c) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 31u) == 0) {
            if (*c.abort_flag) return false;
            if (global_timer_ns() - t0 > c.limit_ns) {
                *c.abort_flag = 1;
                if (c.peer_abort) st_shared_remote(c.peer_abort, 1u);
                atomicOr(c.status, FP8G_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

// All lanes wait; the warp gives up together if any lane gave up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Ctl& c) {
    const bool ok = wait_phase(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait used only while draining at exit (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > DRAIN_LIMIT_NS) break;
}

// After an abort, give asynchronous work still in flight (copies, MMAs and
// the barrier arrivals they trigger) time to land before shared and tensor
// memory are released.
__device__ __forceinline__ void abort_grace() {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ABORT_GRACE_NS) {
    }
}

// The control roles below keep their per-K-block work on one thread (lane 0):
// a K block is a handful of barrier polls, copies or MMAs, and anything the
// whole warp does in that loop (converging, voting) delays the next MMA.  The
// warp only acts together per tile, where the grouped scheduler needs it.

template <int FORM, bool PAIR>
__device__ __forceinline__ void run_producer(const CUtensorMap* map_a, const CUtensorMap* map_b,
                                             const Params& p, int rank, uint8_t* sA, uint8_t* sB,
                                             uint64_t* full, uint64_t* empty, const Ctl& ctl) {
    using C = Cfg<PAIR, FORM>;
    const int lane = threadIdx.x & 31;
    Scheduler<FORM, PAIR> sched(p, rank);
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    for (int t = tile_first<PAIR>(); ok; t += tile_stride<PAIR>()) {
        Tile tile;
        if (!sched.next(t, tile, lane == 0)) break;
        if (tile.skip) continue;
        if (lane == 0) {
            for (int kb = 0; kb < p.kblocks; ++kb) {
                if (!wait_phase(empty + stage, phase ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full + stage, C::STAGE_BYTES);
                tma_load_2d(sA + stage * C::A_BYTES, map_a, full + stage, kb * BLOCK_K, tile.row0);
                tma_load_2d(sB + stage * C::B_BYTES, map_b, full + stage, kb * BLOCK_K,
                            tile.b_row0);
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
    // Every copy issued must have landed before shared memory is released.  (In
    // the even CTA of a pair the phase also needs the odd CTA's relay, which has
    // arrived whenever the pipeline ran to its end.)
    if (lane == 0)
        for (int s = 0; s < C::STAGES; ++s)
            if ((armed >> s) & 1u) drain_wait(full + s, (armed_parity >> s) & 1u);
    __syncwarp();
}

// MMA issuers of a single CTA, or of the even CTA of a pair.  The tensor pipe
// accepts an MMA only when the previous one is under way, so an issuing thread
// is held for most of a K block.  Two warps therefore share the work: the warp
// with `parity` 0 issues the even K blocks (TMEM buffer 0), parity 1 the odd
// ones (buffer 1); while one is held issuing block j, the other has passed the
// barriers of block j+1 and queues it right behind.  A commit tracks only its
// own thread's MMAs, so each block is still signalled exactly when it is done.
template <int FORM, bool PAIR>
__device__ __forceinline__ void run_mma(const Params& p, uint8_t* sA, uint8_t* sB, uint64_t* full,
                                        uint64_t* empty, uint64_t* acc_full, uint64_t* acc_empty,
                                        uint64_t* drain, uint32_t tmem_base, const Ctl& ctl,
                                        int parity) {
    using C = Cfg<PAIR, FORM>;
    const int lane = threadIdx.x & 31;
    Scheduler<FORM, PAIR> sched(p, 0);
    // descriptors of slot 0; slot s is 16-byte units further on
    const uint64_t a_desc0 = smem_desc_k_sw128(smem_u32(sA));
    const uint64_t b_desc0 = smem_desc_k_sw128(smem_u32(sB));
    const int buf = parity;
    const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BLOCK_N);
    uint32_t j = 0;  // K blocks of this CTA's tiles so far, both parities
    bool ok = true;
    for (int t = tile_first<PAIR>(); ok; t += tile_stride<PAIR>()) {
        Tile tile;
        if (!sched.next(t, tile, false)) break;
        if (tile.skip) continue;
        if (lane == 0) {
            for (int kb = 0; kb < p.kblocks; ++kb, ++j) {
                if ((j & 1u) != static_cast<uint32_t>(parity)) continue;
                const uint32_t stage = j % C::STAGES;
                const uint32_t phase = (j / C::STAGES) & 1u;
                const uint32_t bphase = (j >> 1) & 1u;
                if (!wait_phase(acc_empty + buf, bphase ^ 1u, ctl) ||
                    !wait_phase(full + stage, phase, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * C::A_BYTES) >> 4);
                const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * C::B_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < BLOCK_K / UMMA_K; ++kk) {
                    // advance the start address by kk * 32 bytes inside the swizzled rows
                    const uint64_t step = static_cast<uint64_t>((kk * UMMA_K) >> 4);
                    if constexpr (PAIR)
                        umma_f8f6f4_pair(d, ad + step, bd + step, C::IDESC, kk > 0 ? 1u : 0u);
                    else
                        umma_f8f6f4(d, ad + step, bd + step, C::IDESC, kk > 0 ? 1u : 0u);
                }
                if constexpr (PAIR) {
                    umma_commit_pair_multicast(empty + stage, 0x3);   // both CTAs' slots free
                    umma_commit_pair_multicast(acc_full + buf, 0x3);  // both halves ready
                } else {
                    umma_commit(empty + stage);   // smem slot free once these MMAs finish
                    umma_commit(acc_full + buf);  // partial ready for promotion
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    // All MMAs issued must have completed before TMEM and shared memory go away
    // (the drain barrier counts both issuing warps).
    if (lane == 0) {
        if constexpr (PAIR)
            umma_commit_pair(drain);
        else
            umma_commit(drain);
        drain_wait(drain, 0);
    }
    __syncwarp();
}

// Odd CTA of a pair: tell the even CTA each time one of this CTA's slots has
// landed, so that its MMA warp sees both halves of a stage on one barrier.
template <int FORM>
__device__ __forceinline__ void run_relay(const Params& p, uint64_t* full, const Ctl& ctl) {
    using C = Cfg<true, FORM>;
    const int lane = threadIdx.x & 31;
    Scheduler<FORM, true> sched(p, 1);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    uint32_t remote_full[C::STAGES];
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) remote_full[s] = mapa_shared(full + s, 0);
    for (int t = tile_first<true>(); ok; t += tile_stride<true>()) {
        Tile tile;
        if (!sched.next(t, tile, false)) break;
        if (lane == 0) {
            for (int kb = 0; kb < p.kblocks; ++kb) {
                if (!wait_phase(full + stage, phase, ctl)) {
                    ok = false;
                    break;
                }
                mbar_arrive_remote(remote_full[stage]);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, __nv_bfloat16*) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __half*) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
// Four E4M3 codes (first value in the low byte) of v * inv, rounded to nearest
// even and saturated to +-448.
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d, float inv) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a * inv, b * inv), __NV_SATFINITE,
                                                 __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c * inv, d * inv), __NV_SATFINITE,
                                                 __NV_E4M3);
    return lo | (hi << 16);
}

// Epilogue of one promotion warpgroup: its 128 rows x 128 columns of FP32
// sums (thread r holds row r; acc[i] = columns 2i, 2i+1) go out in 128-byte
// row segments: two passes of 64 columns for BF16/FP16, one pass of 128
// columns for E4M3 codes (of value * out_inv).  Each thread rounds its row segment into 128 bytes of shared
// memory (16-byte chunk c of row r at chunk c ^ (r % 8), so that the 32 rows
// a warp writes at once spread over all banks); then each warp stores the 32
// rows it owns as full 128-byte segments, four rows per instruction, skipping
// rows outside the form.  `row_base` is the output row of tile row 0; `cols`
// (a multiple of 16 / sizeof(OutT)) the columns from col0 that exist.
template <typename OutT>
__device__ __forceinline__ void store_tile_rows(OutT* out, int64_t n, int64_t row_base, int col0,
                                                bool row_ok, const uint64_t (&acc)[64],
                                                uint8_t* staging, uint32_t barrier_id,
                                                float out_inv, int cols = 128) {
    constexpr int ESZ = static_cast<int>(sizeof(OutT));  // 2 (BF16/FP16) or 1 (E4M3)
    constexpr int PASSES = ESZ;                          // 128 columns x ESZ bytes
    constexpr int PASS_COLS = 128 / ESZ;
    const int lane = threadIdx.x & 31;
    const int quarter = (threadIdx.x >> 5) & 3;
    const int r = quarter * 32 + lane;
    const uint32_t base = smem_u32(staging);
    OutT* tag = nullptr;
    (void)tag;
    (void)out_inv;
#pragma unroll
    for (int pass = 0; pass < PASSES; ++pass) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 v;
            if constexpr (ESZ == 2) {
                const int a = pass * 32 + 4 * c;  // 8 values
                v.x = pack2(lo_f32(acc[a + 0]), hi_f32(acc[a + 0]), tag);
                v.y = pack2(lo_f32(acc[a + 1]), hi_f32(acc[a + 1]), tag);
                v.z = pack2(lo_f32(acc[a + 2]), hi_f32(acc[a + 2]), tag);
                v.w = pack2(lo_f32(acc[a + 3]), hi_f32(acc[a + 3]), tag);
            } else {
                const int a = 8 * c;  // 16 values
                v.x = pack4_e4m3(lo_f32(acc[a + 0]), hi_f32(acc[a + 0]), lo_f32(acc[a + 1]),
                                 hi_f32(acc[a + 1]), out_inv);
                v.y = pack4_e4m3(lo_f32(acc[a + 2]), hi_f32(acc[a + 2]), lo_f32(acc[a + 3]),
                                 hi_f32(acc[a + 3]), out_inv);
                v.z = pack4_e4m3(lo_f32(acc[a + 4]), hi_f32(acc[a + 4]), lo_f32(acc[a + 5]),
                                 hi_f32(acc[a + 5]), out_inv);
                v.w = pack4_e4m3(lo_f32(acc[a + 6]), hi_f32(acc[a + 6]), lo_f32(acc[a + 7]),
                                 hi_f32(acc[a + 7]), out_inv);
            }
            st_shared_v4(base + r * 128 + ((c ^ (r & 7)) << 4), v);
        }
        named_barrier_sync(barrier_id, 128);
        const int chunk = lane & 7;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = 4 * k + (lane >> 3);  // row within this warp's 32
            const int rr = quarter * 32 + i;    // row within the tile
            const bool ok_i = __shfl_sync(0xffffffffu, row_ok ? 1 : 0, i) != 0;
            const uint4 v = ld_shared_v4(base + rr * 128 + ((chunk ^ (rr & 7)) << 4));
            const int col = pass * PASS_COLS + chunk * (16 / ESZ);
            if (ok_i && col < cols)
                *reinterpret_cast<uint4*>(out + (row_base + rr) * n + col0 + col) = v;
        }
        named_barrier_sync(barrier_id, 128);  // staging free for the next pass
    }
}

// Rounds one promotion thread's row (thread r holds row r of its warpgroup;
// acc[i] = columns 2i, 2i+1) into the warpgroup's tile staging: 128-byte rows,
// 16-byte chunk c of row r at chunk c ^ (r % 8) so that the 32 rows a warp
// writes at once, and the 4 rows the storer reads at once, spread over all
// banks.  BF16/FP16: slice 0 holds columns 0-63, slice 1 columns 64-127;
// E4M3: slice 0 holds the codes of value * out_inv of all 128 columns.
template <typename OutT>
__device__ __forceinline__ void stage_tile_row(uint8_t* staging, const uint64_t (&acc)[64],
                                               float out_inv) {
    constexpr int ESZ = static_cast<int>(sizeof(OutT));
    const int r = ((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31);
    const uint32_t base = smem_u32(staging) + r * 128;
    OutT* tag = nullptr;
    (void)tag;
    (void)out_inv;
#pragma unroll
    for (int slice = 0; slice < ESZ; ++slice) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 v;
            if constexpr (ESZ == 2) {
                const int a = slice * 32 + 4 * c;  // 8 values
                v.x = pack2(lo_f32(acc[a + 0]), hi_f32(acc[a + 0]), tag);
                v.y = pack2(lo_f32(acc[a + 1]), hi_f32(acc[a + 1]), tag);
                v.z = pack2(lo_f32(acc[a + 2]), hi_f32(acc[a + 2]), tag);
                v.w = pack2(lo_f32(acc[a + 3]), hi_f32(acc[a + 3]), tag);
            } else {
                const int a = 8 * c;  // 16 values
                v.x = pack4_e4m3(lo_f32(acc[a + 0]), hi_f32(acc[a + 0]), lo_f32(acc[a + 1]),
                                 hi_f32(acc[a + 1]), out_inv);
                v.y = pack4_e4m3(lo_f32(acc[a + 2]), hi_f32(acc[a + 2]), lo_f32(acc[a + 3]),
                                 hi_f32(acc[a + 3]), out_inv);
                v.z = pack4_e4m3(lo_f32(acc[a + 4]), hi_f32(acc[a + 4]), lo_f32(acc[a + 5]),
                                 hi_f32(acc[a + 5]), out_inv);
                v.w = pack4_e4m3(lo_f32(acc[a + 6]), hi_f32(acc[a + 6]), lo_f32(acc[a + 7]),
                                 hi_f32(acc[a + 7]), out_inv);
            }
            st_shared_v4(base + slice * STAGE_SLICE_BYTES + ((c ^ (r & 7)) << 4), v);
        }
    }
}

// What a promotion warpgroup hands the storer with each staged tile share.
struct StageDesc {
    int32_t x[2];          // per half: first output column of the share
    int32_t y[2];          // per half: output row of tile row 0 (2-D view of out), or
                           // STAGE_END once the warpgroup has no more tiles
    uint32_t row_mask[8];  // [half][quarter]: bit L = row 32 quarter + L is stored
};
constexpr int32_t STAGE_END = -1;

// Warp 3: serves the two promotion warpgroups in turn, one staged tile share
// at a time, and hands the staging back.  A share whose 128 rows are all
// stored goes out as one bulk tensor store per 128-byte column slice
// (`map_out_tile`: 128-row boxes); otherwise every 8-row group whose rows are
// all stored goes out as one (`map_out`: 8-row boxes, the staging's 1 KB
// swizzle atoms), and the rows of the other groups that belong to the form are
// stored by the warp, four 128-byte row segments per instruction.  Lane 0
// issues the bulk stores.  Both
// warpgroups walk the same tiles, so each stages one share per tile and then
// STAGE_END; the storer stops when both have ended (or on an abort), after its
// bulk stores have completed.
template <typename OutT>
__device__ __forceinline__ void run_storer(const CUtensorMap* map_out,
                                           const CUtensorMap* map_out_tile, OutT* out, int64_t n,
                                           uint8_t* sOut, uint64_t* out_full, uint64_t* out_empty,
                                           const StageDesc* desc, const Ctl& ctl) {
    constexpr int ESZ = static_cast<int>(sizeof(OutT));
    constexpr int SLICE_COLS = 128 / ESZ;  // output columns of one 128-byte row
    const int lane = threadIdx.x & 31;
    const int chunk = lane & 7, sub = lane >> 3;
    const volatile StageDesc* vd = desc;
    uint32_t sphase = 0;  // bit h: parity of the next phase of out_full[h]
    uint32_t live = 3;    // bit h: warpgroup h has not ended
    for (int h = 0; live; h ^= 1) {
        if (!((live >> h) & 1u)) continue;
        if (!warp_wait(out_full + h, (sphase >> h) & 1u, ctl)) break;
        sphase ^= 1u << h;
        const int32_t y0 = vd->y[h];
        if (y0 == STAGE_END) {
            live &= ~(1u << h);
            continue;
        }
        const int32_t x0 = vd->x[h];
        const uint32_t base = smem_u32(sOut + h * TILE_STAGE_BYTES);
        uint32_t groups = 0;  // bit g: rows 8g .. 8g+7 are all stored
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t okm = vd->row_mask[h * 4 + q];
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if (((okm >> (8 * b)) & 0xFFu) == 0xFFu) groups |= 1u << (4 * q + b);
        }
        if (lane == 0) {
            if (groups == 0xFFFFu) {  // every row: one 128-row box per slice
                for (int slice = 0; slice < ESZ; ++slice)
                    tma_store_2d(map_out_tile, base + slice * STAGE_SLICE_BYTES,
                                 x0 + slice * SLICE_COLS, y0);
            } else {
#pragma unroll 1
                for (int g = 0; g < 16; ++g)
                    if ((groups >> g) & 1u)
                        for (int slice = 0; slice < ESZ; ++slice)
                            tma_store_2d(map_out, base + slice * STAGE_SLICE_BYTES + g * 1024,
                                         x0 + slice * SLICE_COLS, y0 + 8 * g);
            }
            bulk_commit_group();
        }
        if (groups != 0xFFFFu) {
            uint8_t* d = reinterpret_cast<uint8_t*>(out + static_cast<int64_t>(y0) * n + x0) +
                         chunk * 16;
            const int64_t row_bytes = n * ESZ;
#pragma unroll 1
            for (int slice = 0; slice < ESZ; ++slice) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    const uint32_t okm = vd->row_mask[h * 4 + q];
#pragma unroll 1
                    for (int j = 0; j < 8; ++j) {
                        const int rr = q * 32 + 4 * j + sub;  // the 4 rows share an 8-row group
                        if ((groups >> (rr >> 3)) & 1u) continue;  // stored in bulk
                        const uint4 v = ld_shared_v4(base + slice * STAGE_SLICE_BYTES + rr * 128 +
                                                     ((chunk ^ (rr & 7)) << 4));
                        if ((okm >> (4 * j + sub)) & 1u)
                            *reinterpret_cast<uint4*>(d + rr * row_bytes + slice * 128) = v;
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_read_all();  // the staging has been read
        __syncwarp();
        if (lane == 0) mbar_arrive(out_empty + h);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

// One scale of K block kb (0 where the row or column block is outside the form).
__device__ __forceinline__ float load_scale(const float* x, int step, int kb) {
    return x ? __ldg(x + static_cast<int64_t>(kb) * step) : 0.0f;
}

// Where a promotion thread finds its scales and its output row in a tile.
struct RowScales {
    const float* sa;       // a_scale of the row at K block 0 (null outside the form)
    const float* sb;       // b_scale of the 128-column block at K block 0 (null outside)
    int sa_step, sb_step;  // floats from one K block to the next
    int64_t out_row;       // row of the 2-D view of out
    bool row_ok;           // the row belongs to the form (is stored)
    bool col_ok;           // the warpgroup's 128 columns exist
};

template <int FORM>
__device__ __forceinline__ RowScales row_scales(const Params& p, const Tile& tile, int r,
                                                int quarter, int half) {
    const int KB = p.kblocks;
    const int jb = tile.nb * (BLOCK_N / 128) + half;  // 128-column scale block
    RowScales x;
    x.col_ok = jb < p.nblocks;
    x.sa = x.sb = nullptr;
    x.sa_step = x.sb_step = 1;
    if constexpr (FORM == FORM_MASKED) {
        const int rin = tile.row0 - tile.group * p.rows + r;  // row within the group
        x.out_row = static_cast<int64_t>(tile.group) * p.rows + rin;
        x.row_ok = rin < tile.group_rows;
        if (rin < p.rows) x.sa = p.a_scale + x.out_row * KB;
        if (x.col_ok) x.sb = p.b_scale + (static_cast<int64_t>(tile.group) * p.nblocks + jb) * KB;
    } else {
        x.out_row = static_cast<int64_t>(tile.row0) + r;
        const bool row_in = x.out_row < p.rows;
        if constexpr (FORM == FORM_GROUPED) {
            x.row_ok = row_in && tile.row_expert[quarter] == tile.group;
            if (row_in) x.sa = p.a_scale + x.out_row * KB;
            if (x.col_ok)
                x.sb = p.b_scale + (static_cast<int64_t>(tile.group) * p.nblocks + jb) * KB;
        } else {
            x.row_ok = row_in;
            if (p.scale_mn_major) {
                if (row_in) x.sa = p.a_scale + x.out_row, x.sa_step = p.rows;
                if (x.col_ok) x.sb = p.b_scale + jb, x.sb_step = p.nblocks;
            } else {
                if (row_in) x.sa = p.a_scale + x.out_row * KB;
                if (x.col_ok) x.sb = p.b_scale + static_cast<int64_t>(jb) * KB;
            }
        }
    }
    return x;
}

// acc += s2 * (this warp's 32 rows x 128 columns of FP32 partial sums at
// taddr), acc[i] holding columns 2i and 2i+1, in chunks of CH columns: the
// load of chunk c+1 is in flight while chunk c is accumulated (a TMEM load
// wait covers every load of the thread, so one is in flight at a time).
// release() runs once the whole partial is in registers, before the last
// chunk's FMAs.
template <int CH, typename Release>
__device__ __forceinline__ void promote_partial(uint64_t (&acc)[64], uint32_t taddr, uint64_t s2,
                                                Release release) {
    constexpr int NC = 128 / CH;   // chunks
    constexpr int PAIRS = CH / 2;  // acc entries per chunk
    uint32_t va[CH], vb[CH];
    tmem_load_cols_async(taddr, va);
    tmem_wait_cols(va);
#pragma unroll
    for (int c = 0; c < NC; c += 2) {
        tmem_load_cols_async(taddr + (c + 1) * CH, vb);
#pragma unroll
        for (int i = 0; i < PAIRS; ++i)
            acc[c * PAIRS + i] = ffma2(va[2 * i], va[2 * i + 1], s2, acc[c * PAIRS + i]);
        tmem_wait_cols(vb);
        if (c + 2 < NC)
            tmem_load_cols_async(taddr + (c + 2) * CH, va);
        else
            release();
#pragma unroll
        for (int i = 0; i < PAIRS; ++i)
            acc[(c + 1) * PAIRS + i] = ffma2(vb[2 * i], vb[2 * i + 1], s2, acc[(c + 1) * PAIRS + i]);
        if (c + 2 < NC) tmem_wait_cols(va);
    }
}

template <int FORM, typename OutT, bool PAIR>
__device__ __forceinline__ void run_promotion(const Params& p, int rank, uint64_t* acc_full,
                                              uint64_t* acc_empty, uint32_t tmem_base,
                                              uint8_t* sOut, uint64_t* out_full,
                                              uint64_t* out_empty, StageDesc* desc,
                                              const Ctl& ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quarter = warp & 3;       // this warp may read TMEM lanes 32*quarter .. +31
    const int half = (warp - FIRST_PROMO_WARP) >> 2;  // which 128 columns of the tile
    const int r = quarter * 32 + lane;  // row of the tile owned by this thread
    const int KB = p.kblocks;
    Scheduler<FORM, PAIR> sched(p, rank);
    // E4M3 output: codes of value / out_scale, computed as value * (1 / out_scale)
    float out_inv = 1.0f;
    if constexpr (sizeof(OutT) == 1) out_inv = __frcp_rn(__ldg(p.out_scale));
    // A pair's TMEM buffers are released on the even CTA, whose MMA warp reuses them.
    uint32_t release0 = 0, release1 = 0;
    if constexpr (PAIR) {
        release0 = mapa_shared(acc_empty + 0, 0);
        release1 = mapa_shared(acc_empty + 1, 0);
    }
    using C = Cfg<PAIR, FORM>;
    int buf = 0;
    uint32_t bphase = 0, ephase = 0;
    uint8_t* staging = sOut + half * C::OUT_BYTES;
    bool aborted = false;
    for (int t = tile_first<PAIR>();; t += tile_stride<PAIR>()) {
        Tile tile;
        if (!sched.next(t, tile, false)) break;
        if (tile.skip) continue;

        const RowScales rs = row_scales<FORM>(p, tile, r, quarter, half);
        const bool col_ok = rs.col_ok, row_ok = rs.row_ok;
        // A warp none of whose 32 rows is stored (the tail of a masked group or
        // of an expert's segment, rows past m) or whose half of the tile has no
        // columns reads nothing from TMEM: it only keeps step with the buffer
        // hand-offs, which leaves the tensor-memory bandwidth to the live warps.
        const bool live = col_ok && __any_sync(0xffffffffu, row_ok);
        const float *sa = live ? rs.sa : nullptr, *sb = live ? rs.sb : nullptr;
        const int sa_step = rs.sa_step, sb_step = rs.sb_step;

        uint64_t acc[64];  // FP32 running sums, two columns per register pair
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0;
        // The scales of block kb+1 are loaded while block kb is processed and
        // multiplied only when used, so that a miss in L1 (MN-major scales
        // start a new line every K block) is not waited for early.
        float xa = load_scale(sa, sa_step, 0), xb = load_scale(sb, sb_step, 0);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
            const float s = xa * xb;
            if (kb + 1 < KB) {
                xa = load_scale(sa, sa_step, kb + 1);
                xb = load_scale(sb, sb_step, kb + 1);
            }
            if (!warp_wait(acc_full + buf, bphase, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            if (!live) {
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_remote(buf == 0 ? release0 : release1);
                    else
                        mbar_arrive(acc_empty + buf);
                }
                if (++buf == 2) {
                    buf = 0;
                    bphase ^= 1u;
                }
                continue;
            }
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(buf * BLOCK_N + half * 128);
            // The dense form reads the partial 32 columns per load (4 KB per
            // warp in flight, measured 3-4% faster than 16 columns); the
            // grouped and masked forms keep 16, as 32 spill their tile state.
            constexpr int CHUNK = FORM == FORM_DENSE ? 32 : 16;
            promote_partial<CHUNK>(acc, taddr, splat2(s), [&] {
                // the whole partial is in registers: hand the buffer back first
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_remote(buf == 0 ? release0 : release1);
                    else
                        mbar_arrive(acc_empty + buf);
                }
            });
            if (++buf == 2) {
                buf = 0;
                bphase ^= 1u;
            }
        }
        if constexpr (!C::STORER) {
            // Every warp of the warpgroup takes part in the epilogue's
            // barriers, also after an abort (then storing nothing); the
            // warpgroup stops together.
            if (col_ok)  // uniform over the warpgroup
                store_tile_rows<OutT>(static_cast<OutT*>(p.out), p.n, rs.out_row - r,
                                      tile.nb * BLOCK_N + half * 128, ok && row_ok, acc, staging,
                                      1 + half, out_inv);
            if (named_barrier_or(1 + half, 128, !ok)) break;
            continue;
        }
        // Stage the rounded row for the storer once it has emptied this
        // warpgroup's previous share (a half without columns stages no rows).
        // After an abort nothing is staged (the storer's wait then ends with
        // the abort); every warp still joins the vote, so the warpgroup stops
        // together.
        if (ok && warp_wait(out_empty + half, ephase ^ 1u, ctl)) {
            if (col_ok) {  // uniform
                stage_tile_row<OutT>(staging, acc, out_inv);
                fence_proxy_async_shared();  // the storer's bulk stores read it
            }
            const uint32_t m = __ballot_sync(0xffffffffu, row_ok && col_ok);
            if (lane == 0) desc->row_mask[half * 4 + quarter] = m;
            if (quarter == 0 && lane == 0) {
                desc->x[half] = tile.nb * BLOCK_N + half * 128;
                desc->y[half] = static_cast<int32_t>(rs.out_row - r);
            }
            mbar_arrive(out_full + half);
        } else {
            ok = false;
        }
        ephase ^= 1u;
        if (named_barrier_or(1 + half, 128, !ok)) {
            aborted = true;
            break;
        }
    }
    // No more tiles: tell the storer (after it has emptied the last share).
    if (C::STORER && !aborted && warp_wait(out_empty + half, ephase ^ 1u, ctl)) {
        if (quarter == 0 && lane == 0) desc->y[half] = STAGE_END;
        mbar_arrive(out_full + half);
    }
}

template <int FORM, typename OutT, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ CUtensorMap map_out,
                const __grid_constant__ CUtensorMap map_out_tile, const Params p) {
    using C = Cfg<PAIR, FORM>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    uint8_t* sOut = sB + C::STAGES * C::B_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::SEG_OFFSET + C::SEG_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* acc_full = empty + C::STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* out_full = acc_empty + 2;  // per warpgroup half: its tile share is staged
    uint64_t* out_empty = out_full + 2;  // per half: the storer has emptied the staging
    uint64_t* drain = out_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    StageDesc* stage_desc = reinterpret_cast<StageDesc*>(abort_flag + 1);

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
            mbar_init(out_full + b, 128);  // every thread of the promotion warpgroup
            mbar_init(out_empty + b, 1);
        }
        mbar_init(drain, 2);  // one commit from each MMA-issuing warp
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
        tma_prefetch_map(&map_out);
        tma_prefetch_map(&map_out_tile);
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
    // Everything above touches only this CTA's own resources, so it may overlap
    // the tail of the previous kernel on the stream (launched with programmatic
    // stream serialization); global memory is read and written only after it.
    grid_dependency_wait();
    grid_launch_dependents();
    if constexpr (FORM == FORM_GROUPED) {
        if (p.seg_raster) {  // every role's scheduler reads the table
            if (warp == 0) build_segments(p, reinterpret_cast<int*>(smem + C::SEG_OFFSET));
            __syncthreads();
        }
    }

    if (warp < FIRST_PROMO_WARP) {
        regs_dec<CONTROL_REGS>();
        if (warp == 0) {
            run_producer<FORM, PAIR>(&map_a, &map_b, p, rank, sA, sB, full, empty, ctl);
        } else if (warp == 1 || warp == 2) {
            if constexpr (PAIR) {
                if (rank == 1) {
                    if (warp == 1) run_relay<FORM>(p, full, ctl);
                } else {
                    run_mma<FORM, true>(p, sA, sB, full, empty, acc_full, acc_empty, drain,
                                        tmem_base, ctl, warp - 1);
                }
            } else {
                run_mma<FORM, false>(p, sA, sB, full, empty, acc_full, acc_empty, drain, tmem_base,
                                     ctl, warp - 1);
            }
        } else if constexpr (C::STORER) {
            run_storer<OutT>(&map_out, &map_out_tile, static_cast<OutT*>(p.out), p.n, sOut,
                             out_full, out_empty, stage_desc, ctl);
        }
    } else {
        regs_inc<PROMO_REGS>();
        run_promotion<FORM, OutT, PAIR>(p, rank, acc_full, acc_empty, tmem_base, sOut, out_full,
                                        out_empty, stage_desc, ctl);
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
