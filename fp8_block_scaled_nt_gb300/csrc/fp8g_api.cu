// C ABI of the FP8 groupwise-scaled NT GEMM: host-side validation, tensor-map
// encoding and launch of the sm_103a kernel (gemm_kernel.cuh).
//
// The three entry points follow the MATE page "FlashInfer Wrapper APIs",
// section GEMM (gemm_fp8_nt_groupwise, group_deepgemm_fp8_nt_groupwise,
// batch_deepgemm_fp8_nt_groupwise).  The calling conventions — caller-owned
// memory, enqueue on the caller's stream without synchronising, status code
// plus a last-error message, nothing thrown across the boundary — follow the
// "flashmla-rs" page, section Design Notes.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "fp8g.h"
#include "fp8g_testing.h"
#include "bmm_kernel.cuh"
#include "gemm_kernel.cuh"
#include "moe.cuh"
#include "norm_quant.cuh"

namespace {

using fp8g::Params;

__device__ unsigned int g_device_status;  // OR of FP8G_DEVICE_* bits, per device

// Fixed scratch of the MoE layer's allocation-free entry point, one per device.
static __device__ __align__(256) uint8_t g_moe_static_scratch[FP8G_MOE_STATIC_SCRATCH_BYTES];

thread_local std::string t_last_error;

// Bound of every pipeline wait of the kernels this thread launches (tests of
// the timeout path shorten it through fp8g_testing_set_wait_limit_ns).
thread_local uint64_t t_wait_limit_ns = fp8g::WAIT_LIMIT_NS;

// Tile shape of this thread's last dense GEMM launch: 1 = CTA pairs, 0 = one
// CTA per tile, -1 = none yet (fp8g_testing_last_gemm_cta_pair).
thread_local int t_last_gemm_pair = -1;

fp8g_status_t fail(fp8g_status_t s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

fp8g_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(FP8G_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
// dense bf16, dense f16 (single CTA), grouped, masked, dense bf16, dense f16 (CTA pair),
// dense E4M3 (single CTA), dense E4M3 (CTA pair), bmm bf16, bmm f16, masked (CTA pair),
// bmm bf16 (CTA pair), bmm f16 (CTA pair)
constexpr int kNumKernels = 13;

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int cc_major = 0, cc_minor = 0;
    int sm_count = 0;
    unsigned int* status = nullptr;
    bool kernel_ready[kNumKernels] = {};
    bool norm_ready = false;
    int norm_ring_ctas = 0;  // resident CTAs per SM of the ring norm kernel at its largest row
    bool moe_ready = false;
    uint8_t* moe_static_scratch = nullptr;  // address of g_moe_static_scratch on this device
    int resident[kNumKernels] = {};  // CTAs (or CTA pairs) of a persistent grid
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Current device, checked to be sm_103 and set up once (status word address,
// tensor-map encoder).
fp8g_status_t device_state(DeviceState** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FP8G_ERR_UNSUPPORTED, "device %d", dev);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& ds = g_devices[dev];
    if (!ds.probed) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        ds.cc_major = prop.major;
        ds.cc_minor = prop.minor;
        ds.sm_count = prop.multiProcessorCount;
        ds.supported = prop.major == 10 && prop.minor == 3;
        if (ds.supported) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_device_status);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
            ds.status = static_cast<unsigned int*>(addr);
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail(FP8G_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        ds.probed = true;
    }
    if (!ds.supported)
        return fail(FP8G_ERR_ARCH, "device %d is sm_%d%d; this library needs sm_103 (GB300)", dev,
                    ds.cc_major, ds.cc_minor);
    *out = &ds;
    return FP8G_OK;
}

// Encoded tensor maps, reused across calls.  A map depends only on the
// arguments of cuTensorMapEncodeTiled below, so an entry with the same key is
// the same map whatever happened to the memory in between.  Direct-mapped on a
// hash of the key; a collision replaces the entry.
struct MapKey {
    const void* base;
    int rank;
    cuuint64_t dims[3];
    cuuint64_t strides[2];
    cuuint32_t box[3];
    int dtype, l2, swizzle;
    bool operator==(const MapKey& o) const {
        if (base != o.base || rank != o.rank || dtype != o.dtype || l2 != o.l2 ||
            swizzle != o.swizzle)
            return false;
        for (int i = 0; i < 3; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
        return strides[0] == o.strides[0] && strides[1] == o.strides[1];
    }
};

constexpr int kMapCacheSlots = 256;
struct MapCacheEntry {
    bool used = false;
    MapKey key{};
    CUtensorMap map{};
};
std::mutex g_map_mutex;
MapCacheEntry g_map_cache[kMapCacheSlots];

size_t map_key_hash(const MapKey& k) {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    const uint64_t parts[12] = {static_cast<uint64_t>(k.rank), k.dims[0], k.dims[1], k.dims[2],
                                k.strides[0], k.strides[1], k.box[0], k.box[1], k.box[2],
                                static_cast<uint64_t>(k.dtype), static_cast<uint64_t>(k.l2),
                                static_cast<uint64_t>(k.swizzle)};
    for (uint64_t v : parts) h = (h ^ v) * 0x100000001B3ull;
    return static_cast<size_t>(h ^ (h >> 29)) % kMapCacheSlots;
}

// Tiled map of rank 2 or 3: `dims` = extents in elements, innermost first;
// `strides` = bytes between consecutive indices of dimensions 1 .. rank-1;
// `box` = the copied tile's extents.  Elements outside the extents read as
// zero.
fp8g_status_t encode_tiled(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                           const cuuint64_t* strides, const cuuint32_t* box,
                           CUtensorMapDataType dtype, CUtensorMapL2promotion l2,
                           CUtensorMapSwizzle swizzle, const char* what) {
    MapKey key{};
    key.base = base;
    key.rank = rank;
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank) key.strides[i] = strides[i];
    }
    key.dtype = static_cast<int>(dtype);
    key.l2 = static_cast<int>(l2);
    key.swizzle = static_cast<int>(swizzle);
    const size_t slot = map_key_hash(key);
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        if (g_map_cache[slot].used && g_map_cache[slot].key == key) {
            *map = g_map_cache[slot].map;
            return FP8G_OK;
        }
    }
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                          key.dims, key.strides, key.box, elem_strides,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, l2,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FP8G_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what,
                    static_cast<int>(r));
    std::lock_guard<std::mutex> lock(g_map_mutex);
    g_map_cache[slot].used = true;
    g_map_cache[slot].key = key;
    g_map_cache[slot].map = *map;
    return FP8G_OK;
}

// 2-D tiled map: `dims` = {inner, outer} elements, `stride` = bytes between
// outer rows, `box` = {inner, outer} elements.
fp8g_status_t encode_2d(CUtensorMap* map, const void* base, const cuuint64_t dims[2],
                        cuuint64_t stride, const cuuint32_t box[2], CUtensorMapDataType dtype,
                        CUtensorMapL2promotion l2, CUtensorMapSwizzle swizzle, const char* what) {
    return encode_tiled(map, base, 2, dims, &stride, box, dtype, l2, swizzle, what);
}

// Row-major E4M3 matrix of `rows` x `k` bytes as a 2-D TMA view, tile
// `box_rows` x 128 bytes, 128-byte swizzle; rows past the end read as zero.
fp8g_status_t encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k,
                         int box_rows, const char* what) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(fp8g::BLOCK_K),
                               static_cast<cuuint32_t>(box_rows)};
    return encode_2d(map, base, dims, static_cast<cuuint64_t>(k), box,
                     CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_SWIZZLE_128B, what);
}

// Row-major output of `rows` x `n` elements of `esz` bytes as a 2-D TMA view for
// bulk stores: boxes of `box_rows` rows x 128 bytes, 128-byte swizzle (the
// layout of the kernel's staging).
fp8g_status_t encode_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t n, int esz,
                             int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(rows)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz),
                               static_cast<cuuint32_t>(box_rows)};
    return encode_2d(map, base, dims, static_cast<cuuint64_t>(n * esz), box,
                     esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_SWIZZLE_128B, "out");
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// Shape checks shared by all forms.
fp8g_status_t check_nk(int64_t n, int64_t k) {
    if (n <= 0 || n % 128)
        return fail(FP8G_ERR_INVALID_ARGUMENT, "n = %lld must be a positive multiple of 128",
                    (long long)n);
    if (k <= 0 || k % 128)
        return fail(FP8G_ERR_INVALID_ARGUMENT, "k = %lld must be a positive multiple of 128",
                    (long long)k);
    if (n > kMaxDim || k > kMaxDim)
        return fail(FP8G_ERR_UNSUPPORTED, "n and k must be < 2^31");
    return FP8G_OK;
}

// Pointer checks shared by all forms (non-empty problems only: an empty
// tensor may have a null data pointer).
fp8g_status_t check_ptrs(const void* a, const void* b, const float* a_scale, const float* b_scale,
                         const void* out) {
    if (!a || !b || !a_scale || !b_scale || !out)
        return fail(FP8G_ERR_INVALID_ARGUMENT, "null pointer among a, b, a_scale, b_scale, out");
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(out, 16))
        return fail(FP8G_ERR_INVALID_ARGUMENT, "a, b and out must be 16-byte aligned");
    if (!aligned(a_scale, 4) || !aligned(b_scale, 4))
        return fail(FP8G_ERR_INVALID_ARGUMENT, "scales must be 4-byte aligned");
    return FP8G_OK;
}

template <int FORM, typename OutT, bool PAIR>
fp8g_status_t launch(DeviceState& ds, int slot, const CUtensorMap& map_a, const CUtensorMap& map_b,
                     const Params& p, int64_t max_tiles, cudaStream_t stream) {
    using C = fp8g::Cfg<PAIR, FORM>;
    auto kernel = fp8g::gemm_kernel<FORM, OutT, PAIR>;
    // The kernel's prologue (barriers, TMEM, tensor-map prefetch) may overlap
    // the previous kernel on the stream; it waits for that kernel's completion
    // (griddepcontrol.wait) before touching global memory.
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = 2;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(fp8g::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attrs;
    cfg.numAttrs = PAIR ? 2 : 1;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!ds.kernel_ready[slot]) {
            // The kernel moves registers between its warpgroups (setmaxnreg); that
            // is only safe if it is launched with exactly the budget it was built
            // for, so check the compiled register count before the first launch.
            cudaFuncAttributes attr;
            cudaError_t e = cudaFuncGetAttributes(&attr, kernel);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
            if (attr.numRegs != static_cast<int>(fp8g::LAUNCH_REGS))
                return fail(FP8G_ERR_UNSUPPORTED,
                            "kernel built with %d registers per thread, expected %u", attr.numRegs,
                            fp8g::LAUNCH_REGS);
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(C::SMEM_BYTES));
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            int resident = ds.sm_count;
            if (PAIR) {
                // persistent grid: as many CTA pairs as can be resident at once
                cudaLaunchConfig_t occ = cfg;
                occ.gridDim = dim3(2, 1, 1);
                occ.attrs = &attrs[1];  // the cluster shape alone
                occ.numAttrs = 1;
                int clusters = 0;
                e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &occ);
                if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
                if (clusters < 1)
                    return fail(FP8G_ERR_UNSUPPORTED, "no CTA pair of this kernel fits an SM pair");
                resident = clusters;
            }
            ds.resident[slot] = resident;
            ds.kernel_ready[slot] = true;
        }
    }
    // the 2-D view of out: rows of all groups (masked form) or of the form
    CUtensorMap map_out, map_out_tile;
    const int64_t out_rows =
        FORM == fp8g::FORM_MASKED ? static_cast<int64_t>(p.num_groups) * p.rows : p.rows;
    fp8g_status_t s = encode_out_map(&map_out, p.out, out_rows, p.n, sizeof(OutT), 8);
    if (s == FP8G_OK)
        s = encode_out_map(&map_out_tile, p.out, out_rows, p.n, sizeof(OutT), fp8g::BLOCK_M);
    if (s != FP8G_OK) return s;
    const int64_t units = max_tiles < ds.resident[slot] ? max_tiles : ds.resident[slot];
    cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? 2 * units : units), 1, 1);
    (void)cudaGetLastError();
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, map_a, map_b, map_out, map_out_tile, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    t_last_error.clear();
    return FP8G_OK;
}

Params base_params(const float* a_scale, const float* b_scale, void* out, int64_t rows, int64_t n,
                   int64_t k, int tile_m = fp8g::BLOCK_M) {
    Params p{};
    p.a_scale = a_scale;
    p.b_scale = b_scale;
    p.out = out;
    p.rows = static_cast<int>(rows);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.kblocks = static_cast<int>(k / 128);
    p.nblocks = static_cast<int>(n / 128);
    p.n_tiles = static_cast<int>((n + fp8g::BLOCK_N - 1) / fp8g::BLOCK_N);
    p.m_blocks = static_cast<int>((rows + tile_m - 1) / tile_m);
    // raster bands of the dense form: 16 m-blocks (measured best of 4-32 on
    // 16384 x 18432 x 7168 and 4096 x 7168 x 2048; the grouped form sets its own)
    p.band_m = 16;
    p.wait_limit_ns = t_wait_limit_ns;
    return p;
}

// bmm_fp8 kernel launch (persistent, one CTA or CTA pair per SM or SM pair) on
// validated arguments.
template <typename OutT, bool PAIR>
fp8g_status_t launch_bmm(DeviceState& ds, int slot, const CUtensorMap& map_a,
                         const CUtensorMap& map_b, const Params& p, int64_t tiles,
                         cudaStream_t stream) {
    using C = fp8g::BmmCfg<PAIR>;
    auto kernel = fp8g::bmm_kernel<OutT, PAIR>;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    attrs[1].id = cudaLaunchAttributeClusterDimension;
    attrs[1].val.clusterDim.x = 2;
    attrs[1].val.clusterDim.y = 1;
    attrs[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(fp8g::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attrs;
    cfg.numAttrs = PAIR ? 2 : 1;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!ds.kernel_ready[slot]) {
            cudaFuncAttributes attr;
            cudaError_t e = cudaFuncGetAttributes(&attr, kernel);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
            if (attr.numRegs != static_cast<int>(fp8g::LAUNCH_REGS))
                return fail(FP8G_ERR_UNSUPPORTED,
                            "kernel built with %d registers per thread, expected %u", attr.numRegs,
                            fp8g::LAUNCH_REGS);
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(C::SMEM_BYTES));
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            int resident = ds.sm_count;
            if (PAIR) {
                cudaLaunchConfig_t occ = cfg;
                occ.gridDim = dim3(2, 1, 1);
                occ.attrs = &attrs[1];  // the cluster shape alone
                occ.numAttrs = 1;
                int clusters = 0;
                e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &occ);
                if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
                if (clusters < 1)
                    return fail(FP8G_ERR_UNSUPPORTED, "no CTA pair of this kernel fits an SM pair");
                resident = clusters;
            }
            ds.resident[slot] = resident;
            ds.kernel_ready[slot] = true;
        }
    }
    const int64_t units = tiles < ds.resident[slot] ? tiles : ds.resident[slot];
    cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? 2 * units : units), 1, 1);
    (void)cudaGetLastError();
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, map_a, map_b, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return FP8G_OK;
}

// Contiguous grouped GEMM on validated arguments (m > 0).
fp8g_status_t grouped_gemm(DeviceState& ds, const void* a, const void* b, const float* a_scale,
                           const float* b_scale, const int32_t* m_indices, void* out, int64_t m,
                           int64_t n, int64_t k, int64_t num_groups, cudaStream_t stream) {
    const int64_t tiles = ((m + 127) / 128) * ((n + 255) / 256);
    fp8g_status_t s;
    CUtensorMap map_a, map_b;
    if ((s = encode_map(&map_a, a, m, k, fp8g::BLOCK_M, "a")) != FP8G_OK) return s;
    if ((s = encode_map(&map_b, b, num_groups * n, k, fp8g::BLOCK_N, "b")) != FP8G_OK) return s;
    Params p = base_params(a_scale, b_scale, out, m, n, k);
    // tiles ordered by expert segment where the segment table fits; else bands
    // of 4 m-blocks (fewer bands straddle two experts' segments, whose weights
    // then stream twice; measured best of 4-32 on 4096 tokens x top-8 over 64
    // experts)
    p.seg_raster = p.m_blocks <= fp8g::SEG_RASTER_MAX_BLOCKS;
    p.band_m = 4;
    p.num_tiles = static_cast<int>(tiles);
    p.num_groups = static_cast<int>(num_groups);
    p.m_indices = m_indices;
    p.status = ds.status;
    return launch<fp8g::FORM_GROUPED, __nv_bfloat16, false>(ds, 2, map_a, map_b, p, tiles, stream);
}

// Launch of a plain kernel with programmatic stream serialization.
template <typename... KArgs, typename... Args>
fp8g_status_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                         cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    (void)cudaGetLastError();
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return FP8G_OK;
}

// Workspace of the MoE layer: the regions, each 256-byte aligned.
struct MoeWorkspace {
    int64_t rows;  // M
    size_t m_indices, row_of, a1, a1_scale, h, a2, a2_scale, y, total;
};

MoeWorkspace moe_workspace(int64_t tokens, int64_t experts, int64_t top_k, int64_t hidden,
                           int64_t inter) {
    MoeWorkspace w{};
    w.rows = fp8g::moe_rows(tokens, top_k, experts);
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t start = at;
        at += (bytes + 255) / 256 * 256;
        return start;
    };
    const size_t M = static_cast<size_t>(w.rows);
    w.m_indices = take(4 * M);
    w.row_of = take(4 * static_cast<size_t>(tokens * top_k));
    w.a1 = take(M * hidden);
    w.a1_scale = take(4 * M * (hidden / 128));
    w.h = take(2 * M * 2 * inter);
    w.a2 = take(M * inter);
    w.a2_scale = take(4 * M * (inter / 128));
    w.y = take(2 * M * hidden);
    w.total = at;
    return w;
}

fp8g_status_t check_moe_shape(int64_t tokens, int64_t experts, int64_t top_k, int64_t hidden,
                              int64_t inter) {
    if (tokens < 0) return fail(FP8G_ERR_INVALID_ARGUMENT, "num_tokens = %lld < 0", (long long)tokens);
    if (experts <= 0 || experts > fp8g::MOE_MAX_EXPERTS)
        return fail(FP8G_ERR_INVALID_ARGUMENT, "num_experts = %lld must be in [1, %d]",
                    (long long)experts, fp8g::MOE_MAX_EXPERTS);
    if (top_k <= 0 || top_k > experts)
        return fail(FP8G_ERR_INVALID_ARGUMENT, "top_k = %lld must be in [1, num_experts]",
                    (long long)top_k);
    if (hidden <= 0 || hidden % 128)
        return fail(FP8G_ERR_INVALID_ARGUMENT,
                    "hidden_size = %lld must be a positive multiple of 128", (long long)hidden);
    if (inter <= 0 || inter % 128)
        return fail(FP8G_ERR_INVALID_ARGUMENT,
                    "inter_size = %lld must be a positive multiple of 128", (long long)inter);
    const int64_t rows = fp8g::moe_rows(tokens, top_k, experts);
    if (tokens * top_k > kMaxDim || rows > kMaxDim || experts * 2 * inter > kMaxDim ||
        experts * hidden > kMaxDim || rows * 2 * inter > (int64_t(1) << 40))
        return fail(FP8G_ERR_UNSUPPORTED, "MoE problem too large");
    return FP8G_OK;
}

// The MoE layer on validated arguments and a workspace of at least
// moe_workspace(...).total bytes.
fp8g_status_t moe_run(DeviceState& ds, const void* input, const int32_t* token_selected,
                      const void* fc1_weights, const void* fc2_weights, void* out,
                      const float* fc1_scales, const float* fc2_scales, int64_t tokens,
                      int64_t experts, int64_t top_k, int64_t hidden, int64_t inter,
                      uint8_t* ws, cudaStream_t stream) {
    const MoeWorkspace w = moe_workspace(tokens, experts, top_k, hidden, inter);
    int32_t* m_indices = reinterpret_cast<int32_t*>(ws + w.m_indices);
    int32_t* row_of = reinterpret_cast<int32_t*>(ws + w.row_of);
    uint8_t* a1 = ws + w.a1;
    float* a1_scale = reinterpret_cast<float*>(ws + w.a1_scale);
    uint16_t* h = reinterpret_cast<uint16_t*>(ws + w.h);
    uint8_t* a2 = ws + w.a2;
    float* a2_scale = reinterpret_cast<float*>(ws + w.a2_scale);
    uint16_t* y = reinterpret_cast<uint16_t*>(ws + w.y);
    fp8g_status_t s;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!ds.moe_ready) {
            cudaError_t e = cudaFuncSetAttribute(fp8g::moe_route_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 3 * 4 * fp8g::MOE_MAX_EXPERTS);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
            ds.moe_ready = true;
        }
    }
    if ((s = launch_pdl(fp8g::moe_route_kernel, 1, fp8g::MOE_ROUTE_THREADS,
                        static_cast<size_t>(12 * experts), stream, token_selected,
                        static_cast<int>(tokens * top_k), static_cast<int>(experts),
                        static_cast<int>(w.rows), m_indices, row_of, ds.status)) != FP8G_OK)
        return s;
    if ((s = launch_pdl(fp8g::moe_quant_gather_kernel, static_cast<unsigned>(tokens),
                        fp8g::MOE_ROW_THREADS, 0, stream, static_cast<const uint16_t*>(input),
                        static_cast<const int32_t*>(row_of), static_cast<int>(top_k),
                        static_cast<int>(hidden), a1, a1_scale)) != FP8G_OK)
        return s;
    if ((s = grouped_gemm(ds, a1, fc1_weights, a1_scale, fc1_scales, m_indices, h, w.rows,
                          2 * inter, hidden, experts, stream)) != FP8G_OK)
        return s;
    if ((s = launch_pdl(fp8g::moe_swiglu_quant_kernel, static_cast<unsigned>(w.rows),
                        fp8g::MOE_ROW_THREADS, 0, stream, static_cast<const uint16_t*>(h),
                        static_cast<const int32_t*>(m_indices), static_cast<int>(inter), a2,
                        a2_scale)) != FP8G_OK)
        return s;
    if ((s = grouped_gemm(ds, a2, fc2_weights, a2_scale, fc2_scales, m_indices, y, w.rows,
                          hidden, inter, experts, stream)) != FP8G_OK)
        return s;
    return launch_pdl(fp8g::moe_combine_kernel, static_cast<unsigned>(tokens),
                      fp8g::MOE_ROW_THREADS, 0, stream, static_cast<const uint16_t*>(y),
                      static_cast<const int32_t*>(row_of), static_cast<int>(top_k),
                      static_cast<int>(hidden), static_cast<uint16_t*>(out));
}

}  // namespace

extern "C" {

const char* fp8g_last_error(void) { return t_last_error.c_str(); }

fp8g_status_t fp8_gemm_nt_groupwise(const void* a, const void* b, const float* a_scale,
                                    const float* b_scale, void* out, fp8g_dtype_t out_dtype,
                                    const float* output_scale, int64_t m, int64_t n, int64_t k,
                                    fp8g_scale_major_t scale_major,
                                    int gran_m, int gran_n, int gran_k, int mma_sm,
                                    cudaStream_t stream) {
    try {
        if (m < 0) return fail(FP8G_ERR_INVALID_ARGUMENT, "m = %lld < 0", (long long)m);
        if (out_dtype != FP8G_OUT_BF16 && out_dtype != FP8G_OUT_F16 &&
            out_dtype != FP8G_OUT_E4M3)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "out_dtype %d is not BF16, FP16 or E4M3",
                        (int)out_dtype);
        if ((out_dtype == FP8G_OUT_E4M3) != (output_scale != nullptr))
            return fail(FP8G_ERR_INVALID_ARGUMENT,
                        "output_scale must be given exactly when out_dtype is E4M3");
        if (output_scale && !aligned(output_scale, 4))
            return fail(FP8G_ERR_INVALID_ARGUMENT, "output_scale must be 4-byte aligned");
        if (scale_major != FP8G_SCALE_K_MAJOR && scale_major != FP8G_SCALE_MN_MAJOR)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "scale_major %d is neither K nor MN",
                        (int)scale_major);
        if (mma_sm < 0 || mma_sm > 2)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "mma_sm = %d (expected 0, 1 or 2)", mma_sm);
        if (gran_m != 1 || gran_n != 128 || gran_k != 128)
            return fail(FP8G_ERR_UNSUPPORTED,
                        "scale granularity (%d,%d,%d): only (1,128,128) is provided", gran_m,
                        gran_n, gran_k);
        if (m > kMaxDim) return fail(FP8G_ERR_UNSUPPORTED, "m must be < 2^31");
        fp8g_status_t s = check_nk(n, k);
        if (s != FP8G_OK) return s;
        if (m == 0) {
            t_last_error.clear();
            return FP8G_OK;
        }
        if ((s = check_ptrs(a, b, a_scale, b_scale, out)) != FP8G_OK) return s;
        const int64_t n_tiles = (n + 255) / 256;
        if (((m + 127) / 128) * n_tiles > kMaxDim)
            return fail(FP8G_ERR_UNSUPPORTED, "problem has too many tiles");
        DeviceState* ds = nullptr;
        if ((s = device_state(&ds)) != FP8G_OK) return s;
        // mma_sm: 1 = one SM per 128x256 tile, 2 = a CTA pair per 256x256 tile
        // (tcgen05 cta_group::2), 0 = pairs when there are enough 256-row tiles
        // to give every SM pair work.  Results are identical either way.
        const int64_t pair_tiles = ((m + 255) / 256) * n_tiles;
        const bool pair = mma_sm == 2 || (mma_sm == 0 && m > 128 && 2 * pair_tiles >= ds->sm_count);
        const int tile_m = pair ? 2 * fp8g::BLOCK_M : fp8g::BLOCK_M;
        const int64_t tiles = ((m + tile_m - 1) / tile_m) * n_tiles;
        CUtensorMap map_a, map_b;
        if ((s = encode_map(&map_a, a, m, k, fp8g::BLOCK_M, "a")) != FP8G_OK) return s;
        if ((s = encode_map(&map_b, b, n, k, pair ? fp8g::BLOCK_N / 2 : fp8g::BLOCK_N, "b")) !=
            FP8G_OK)
            return s;
        Params p = base_params(a_scale, b_scale, out, m, n, k, tile_m);
        t_last_gemm_pair = pair ? 1 : 0;
        p.num_tiles = static_cast<int>(tiles);
        p.num_groups = 1;
        p.scale_mn_major = scale_major == FP8G_SCALE_MN_MAJOR;
        p.out_scale = output_scale;
        p.status = ds->status;
        if (out_dtype == FP8G_OUT_E4M3)
            return pair ? launch<fp8g::FORM_DENSE, __nv_fp8_e4m3, true>(*ds, 7, map_a, map_b, p,
                                                                        tiles, stream)
                        : launch<fp8g::FORM_DENSE, __nv_fp8_e4m3, false>(*ds, 6, map_a, map_b, p,
                                                                         tiles, stream);
        if (out_dtype == FP8G_OUT_BF16)
            return pair ? launch<fp8g::FORM_DENSE, __nv_bfloat16, true>(*ds, 4, map_a, map_b, p,
                                                                        tiles, stream)
                        : launch<fp8g::FORM_DENSE, __nv_bfloat16, false>(*ds, 0, map_a, map_b, p,
                                                                         tiles, stream);
        return pair ? launch<fp8g::FORM_DENSE, __half, true>(*ds, 5, map_a, map_b, p, tiles, stream)
                    : launch<fp8g::FORM_DENSE, __half, false>(*ds, 1, map_a, map_b, p, tiles,
                                                              stream);
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

fp8g_status_t fp8_group_gemm_contiguous(const void* a, const void* b, const float* a_scale,
                                        const float* b_scale, const int32_t* m_indices, void* out,
                                        int64_t m, int64_t n, int64_t k, int64_t num_groups,
                                        cudaStream_t stream) {
    try {
        if (m < 0) return fail(FP8G_ERR_INVALID_ARGUMENT, "m = %lld < 0", (long long)m);
        if (num_groups <= 0)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "num_groups = %lld must be >= 1",
                        (long long)num_groups);
        if (m > kMaxDim) return fail(FP8G_ERR_UNSUPPORTED, "m must be < 2^31");
        fp8g_status_t s = check_nk(n, k);
        if (s != FP8G_OK) return s;
        if (num_groups * n > kMaxDim)
            return fail(FP8G_ERR_UNSUPPORTED, "num_groups * n must be < 2^31");
        if (m == 0) {
            t_last_error.clear();
            return FP8G_OK;
        }
        if ((s = check_ptrs(a, b, a_scale, b_scale, out)) != FP8G_OK) return s;
        if (!m_indices) return fail(FP8G_ERR_INVALID_ARGUMENT, "m_indices is null");
        if (!aligned(m_indices, 4))
            return fail(FP8G_ERR_INVALID_ARGUMENT, "m_indices must be 4-byte aligned");
        const int64_t tiles = ((m + 127) / 128) * ((n + 255) / 256);
        if (tiles > kMaxDim) return fail(FP8G_ERR_UNSUPPORTED, "problem has too many tiles");
        DeviceState* ds = nullptr;
        if ((s = device_state(&ds)) != FP8G_OK) return s;
        return grouped_gemm(*ds, a, b, a_scale, b_scale, m_indices, out, m, n, k, num_groups,
                            stream);
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

fp8g_status_t fp8_batch_gemm_masked(const void* a, const void* b, const float* a_scale,
                                    const float* b_scale, const int32_t* masked_m,
                                    int64_t expected_m, void* out, int64_t num_groups,
                                    int64_t max_m, int64_t n, int64_t k, cudaStream_t stream) {
    try {
        if (num_groups < 0 || max_m < 0)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "num_groups = %lld and max_m = %lld must be >= 0",
                        (long long)num_groups, (long long)max_m);
        if (expected_m < 0)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "expected_m = %lld < 0", (long long)expected_m);
        fp8g_status_t s = check_nk(n, k);
        if (s != FP8G_OK) return s;
        if (num_groups * max_m > kMaxDim || num_groups * n > kMaxDim)
            return fail(FP8G_ERR_UNSUPPORTED, "num_groups * max_m and num_groups * n must be < 2^31");
        const int64_t tiles = num_groups * ((max_m + 127) / 128) * ((n + 255) / 256);
        if (tiles > kMaxDim) return fail(FP8G_ERR_UNSUPPORTED, "problem has too many tiles");
        if (tiles == 0) {
            t_last_error.clear();
            return FP8G_OK;
        }
        if ((s = check_ptrs(a, b, a_scale, b_scale, out)) != FP8G_OK) return s;
        if (!masked_m) return fail(FP8G_ERR_INVALID_ARGUMENT, "masked_m is null");
        if (!aligned(masked_m, 4))
            return fail(FP8G_ERR_INVALID_ARGUMENT, "masked_m must be 4-byte aligned");
        DeviceState* ds = nullptr;
        if ((s = device_state(&ds)) != FP8G_OK) return s;
        // expected_m (the page's kernel-selection hint) picks the tile shape:
        // when a typical group holds more than 128 rows, CTA pairs compute 256-row
        // tiles (a third less operand traffic per SM); otherwise one CTA per
        // 128-row tile, which wastes less on short groups.  Results are the same
        // bits either way.
        const bool pair = expected_m > fp8g::BLOCK_M && max_m > fp8g::BLOCK_M;
        const int tile_m = pair ? 2 * fp8g::BLOCK_M : fp8g::BLOCK_M;
        const int64_t max_tiles = num_groups * ((max_m + tile_m - 1) / tile_m) * ((n + 255) / 256);
        CUtensorMap map_a, map_b;
        if ((s = encode_map(&map_a, a, num_groups * max_m, k, fp8g::BLOCK_M, "a")) != FP8G_OK)
            return s;
        if ((s = encode_map(&map_b, b, num_groups * n, k,
                            pair ? fp8g::BLOCK_N / 2 : fp8g::BLOCK_N, "b")) != FP8G_OK)
            return s;
        Params p = base_params(a_scale, b_scale, out, max_m, n, k, tile_m);
        p.num_tiles = static_cast<int>(max_tiles);  // upper bound; the kernel walks masked_m
        p.num_groups = static_cast<int>(num_groups);
        p.masked_m = masked_m;
        p.status = ds->status;
        if (pair)
            return launch<fp8g::FORM_MASKED, __nv_bfloat16, true>(*ds, 10, map_a, map_b, p,
                                                                  max_tiles, stream);
        return launch<fp8g::FORM_MASKED, __nv_bfloat16, false>(*ds, 3, map_a, map_b, p, max_tiles,
                                                                stream);
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

fp8g_status_t fused_add_rmsnorm_fp8_block_quant(void* out, float* block_scale, void* normed_out,
                                                const void* input, void* residual,
                                                const void* weight, float eps, int64_t rows,
                                                int64_t hidden, cudaStream_t stream) {
    try {
        if (rows < 0) return fail(FP8G_ERR_INVALID_ARGUMENT, "rows = %lld < 0", (long long)rows);
        if (hidden <= 0 || hidden % 128)
            return fail(FP8G_ERR_INVALID_ARGUMENT,
                        "hidden = %lld must be a positive multiple of 128", (long long)hidden);
        if (hidden > 65536)
            return fail(FP8G_ERR_UNSUPPORTED, "hidden = %lld > 65536", (long long)hidden);
        if (!(eps >= 0.0f) || !std::isfinite(eps))
            return fail(FP8G_ERR_INVALID_ARGUMENT, "eps must be finite and >= 0");
        if (rows > kMaxDim) return fail(FP8G_ERR_UNSUPPORTED, "rows must be < 2^31");
        if (rows == 0) {
            t_last_error.clear();
            return FP8G_OK;
        }
        if (!out || !block_scale || !normed_out || !input || !residual || !weight)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "null pointer argument");
        if (!aligned(out, 16) || !aligned(normed_out, 16) || !aligned(input, 16) ||
            !aligned(residual, 16) || !aligned(weight, 16) || !aligned(block_scale, 4))
            return fail(FP8G_ERR_INVALID_ARGUMENT,
                        "out, normed_out, input, residual and weight must be 16-byte aligned, "
                        "block_scale 4-byte aligned");
        DeviceState* ds = nullptr;
        fp8g_status_t s = device_state(&ds);
        if (s != FP8G_OK) return s;
        // rows of up to NQR_MAX_HIDDEN: the persistent kernel with the bulk-copy
        // ring; longer rows: one CTA per row
        const bool ring = hidden <= fp8g::NQR_MAX_HIDDEN;
        const size_t ring_max_smem =
            static_cast<size_t>(fp8g::NQR_STAGES) * 4 * fp8g::NQR_MAX_HIDDEN;
        {
            std::lock_guard<std::mutex> lock(g_mutex);
            if (!ds->norm_ready) {
                cudaError_t e = cudaFuncSetAttribute(fp8g::fused_add_rmsnorm_quant_kernel,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     65536 * 2);
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(fp8g::fused_add_rmsnorm_quant_ring_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(ring_max_smem));
                if (e == cudaSuccess)
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &ds->norm_ring_ctas, fp8g::fused_add_rmsnorm_quant_ring_kernel,
                        fp8g::NQ_THREADS, ring_max_smem);
                if (e != cudaSuccess) return cuda_fail(e, "norm kernel attributes");
                if (ds->norm_ring_ctas < 1) ds->norm_ring_ctas = 1;
                ds->norm_ready = true;
            }
        }
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(fp8g::NQ_THREADS, 1, 1);
        cfg.stream = stream;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        (void)cudaGetLastError();
        cudaError_t e;
        if (ring) {
            const int64_t grid = std::min<int64_t>(rows, int64_t(ds->sm_count) * ds->norm_ring_ctas);
            cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
            cfg.dynamicSmemBytes = static_cast<size_t>(fp8g::NQR_STAGES) * 4 * hidden;
            e = cudaLaunchKernelEx(&cfg, fp8g::fused_add_rmsnorm_quant_ring_kernel,
                                   static_cast<uint8_t*>(out), block_scale,
                                   static_cast<uint16_t*>(normed_out),
                                   static_cast<const uint16_t*>(input),
                                   static_cast<uint16_t*>(residual),
                                   static_cast<const uint16_t*>(weight), eps,
                                   static_cast<int>(rows), static_cast<int>(hidden), ds->status);
        } else {
            cfg.gridDim = dim3(static_cast<unsigned>(rows), 1, 1);
            cfg.dynamicSmemBytes = static_cast<size_t>(hidden) * 2;
            e = cudaLaunchKernelEx(&cfg, fp8g::fused_add_rmsnorm_quant_kernel,
                                   static_cast<uint8_t*>(out), block_scale,
                                   static_cast<uint16_t*>(normed_out),
                                   static_cast<const uint16_t*>(input),
                                   static_cast<uint16_t*>(residual),
                                   static_cast<const uint16_t*>(weight), eps,
                                   static_cast<int>(rows), static_cast<int>(hidden));
        }
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
        t_last_error.clear();
        return FP8G_OK;
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

fp8g_status_t bmm_fp8(const void* a, const void* b, fp8g_fp8_format_t a_format,
                      fp8g_fp8_format_t b_format, const float* a_scale, int a_channelwise,
                      const float* b_scale, int b_channelwise, void* out,
                      fp8g_dtype_t out_dtype, int64_t batch, int64_t m, int64_t n, int64_t k,
                      cudaStream_t stream) {
    try {
        if (batch < 0 || m < 0)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "batch = %lld and m = %lld must be >= 0",
                        (long long)batch, (long long)m);
        if ((a_format != FP8G_FP8_E4M3 && a_format != FP8G_FP8_E5M2) ||
            (b_format != FP8G_FP8_E4M3 && b_format != FP8G_FP8_E5M2))
            return fail(FP8G_ERR_INVALID_ARGUMENT, "operand formats must be E4M3 or E5M2");
        if (out_dtype != FP8G_OUT_BF16 && out_dtype != FP8G_OUT_F16)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "out_dtype %d is neither BF16 nor FP16",
                        (int)out_dtype);
        // n and k need only be multiples of 16: TMA views want 16-byte row
        // pitches; the tails of the last 128-wide blocks read as zero.
        if (n <= 0 || n % 16)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "n = %lld must be a positive multiple of 16",
                        (long long)n);
        if (k <= 0 || k % 16)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "k = %lld must be a positive multiple of 16",
                        (long long)k);
        fp8g_status_t s = FP8G_OK;
        if (n > kMaxDim || k > kMaxDim || batch * m > kMaxDim || batch * n > kMaxDim)
            return fail(FP8G_ERR_UNSUPPORTED, "n, k, batch * m and batch * n must be < 2^31");
        const int64_t m_blocks = (m + 127) / 128, n_tiles = (n + 255) / 256;
        const int64_t tiles = batch * m_blocks * n_tiles;
        if (tiles > kMaxDim) return fail(FP8G_ERR_UNSUPPORTED, "problem has too many tiles");
        if (tiles == 0) {
            t_last_error.clear();
            return FP8G_OK;
        }
        if ((s = check_ptrs(a, b, a_scale, b_scale, out)) != FP8G_OK) return s;
        DeviceState* ds = nullptr;
        if ((s = device_state(&ds)) != FP8G_OK) return s;
        CUtensorMap map_a, map_b;
        // A: (batch * m) rows of k; a K block past k reads zeros.  A tile's rows
        // past m belong to the next batch (or read as zero); they are not stored.
        if ((s = encode_map(&map_a, a, batch * m, k, fp8g::BLOCK_M, "a")) != FP8G_OK) return s;
        // B stays N-major, as a 3-D view (n, k, batch) in boxes of 128 columns x
        // 128 k-rows of one batch: k-rows past k read as zero rather than as the
        // next batch's rows, so no value of another batch (an infinity or NaN
        // of E5M2) meets the zeros of A's tail.
        {
            const cuuint64_t dims[3] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(k),
                                        static_cast<cuuint64_t>(batch)};
            const cuuint64_t strides[2] = {static_cast<cuuint64_t>(n),
                                           static_cast<cuuint64_t>(n) * static_cast<cuuint64_t>(k)};
            const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(fp8g::BLOCK_K), 1};
            if ((s = encode_tiled(&map_b, b, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_SWIZZLE_128B,
                                  "b")) != FP8G_OK)
                return s;
        }
        // CTA pairs on 256 x 256 tiles when there are enough of them to give every
        // SM pair work (results are identical either way)
        const int64_t pair_tiles = batch * ((m + 255) / 256) * n_tiles;
        const bool pair = m > 128 && 2 * pair_tiles >= ds->sm_count;
        const int tile_m = pair ? 2 * fp8g::BLOCK_M : fp8g::BLOCK_M;
        const int64_t launch_tiles = pair ? pair_tiles : tiles;
        Params p = base_params(a_scale, b_scale, out, m, n, k, tile_m);
        p.kblocks = static_cast<int>((k + fp8g::BLOCK_K - 1) / fp8g::BLOCK_K);
        p.band_m = 8;
        p.num_tiles = static_cast<int>(launch_tiles);
        p.batch = static_cast<int>(batch);
        p.a_channelwise = a_channelwise != 0;
        p.b_channelwise = b_channelwise != 0;
        p.idesc = fp8g::idesc_bmm(static_cast<uint32_t>(a_format), static_cast<uint32_t>(b_format),
                                  static_cast<uint32_t>(tile_m));
        p.status = ds->status;
        t_last_gemm_pair = pair ? 1 : 0;
        if (out_dtype == FP8G_OUT_BF16)
            return pair ? launch_bmm<__nv_bfloat16, true>(*ds, 11, map_a, map_b, p, launch_tiles,
                                                           stream)
                        : launch_bmm<__nv_bfloat16, false>(*ds, 8, map_a, map_b, p, launch_tiles,
                                                            stream);
        return pair ? launch_bmm<__half, true>(*ds, 12, map_a, map_b, p, launch_tiles, stream)
                    : launch_bmm<__half, false>(*ds, 9, map_a, map_b, p, launch_tiles, stream);
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

size_t fused_moe_deepseek_fp8_block_scale_workspace_size(int64_t num_tokens, int64_t num_experts,
                                                         int64_t top_k, int64_t hidden_size,
                                                         int64_t inter_size) {
    if (check_moe_shape(num_tokens, num_experts, top_k, hidden_size, inter_size) != FP8G_OK)
        return 0;
    return moe_workspace(num_tokens, num_experts, top_k, hidden_size, inter_size).total;
}

fp8g_status_t fused_moe_deepseek_fp8_block_scale(
    const void* input, const int32_t* token_selected, const void* fc1_weights,
    const void* fc2_weights, void* out, const float* fc1_scales, const float* fc2_scales,
    int64_t num_tokens, int64_t num_experts, int64_t top_k, int64_t hidden_size,
    int64_t inter_size, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    try {
        fp8g_status_t s = check_moe_shape(num_tokens, num_experts, top_k, hidden_size,
                                          inter_size);
        if (s != FP8G_OK) return s;
        if (num_tokens == 0) {
            t_last_error.clear();
            return FP8G_OK;
        }
        if (!input || !token_selected || !fc1_weights || !fc2_weights || !out || !fc1_scales ||
            !fc2_scales || !workspace)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "null pointer argument");
        if (!aligned(input, 16) || !aligned(fc1_weights, 16) || !aligned(fc2_weights, 16) ||
            !aligned(out, 16) || !aligned(workspace, 256) || !aligned(token_selected, 4) ||
            !aligned(fc1_scales, 4) || !aligned(fc2_scales, 4))
            return fail(FP8G_ERR_INVALID_ARGUMENT,
                        "input, weights and out must be 16-byte aligned, workspace 256-byte "
                        "aligned, token_selected and scales 4-byte aligned");
        const size_t need =
            moe_workspace(num_tokens, num_experts, top_k, hidden_size, inter_size).total;
        if (workspace_bytes < need)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "workspace of %zu bytes, %zu needed",
                        workspace_bytes, need);
        DeviceState* ds = nullptr;
        if ((s = device_state(&ds)) != FP8G_OK) return s;
        s = moe_run(*ds, input, token_selected, fc1_weights, fc2_weights, out, fc1_scales,
                    fc2_scales, num_tokens, num_experts, top_k, hidden_size, inter_size,
                    static_cast<uint8_t*>(workspace), stream);
        if (s == FP8G_OK) t_last_error.clear();
        return s;
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

fp8g_status_t fused_moe_deepseek_fp8_block_scale_noalloc(
    const void* input, const int32_t* token_selected, const void* fc1_weights,
    const void* fc2_weights, void* out, const float* fc1_scales, const float* fc2_scales,
    int64_t num_tokens, int64_t num_experts, int64_t top_k, int64_t hidden_size,
    int64_t inter_size, cudaStream_t stream) {
    try {
        fp8g_status_t s = check_moe_shape(num_tokens, num_experts, top_k, hidden_size,
                                          inter_size);
        if (s != FP8G_OK) return s;
        if (num_tokens == 0) {
            t_last_error.clear();
            return FP8G_OK;
        }
        if (!input || !token_selected || !fc1_weights || !fc2_weights || !out || !fc1_scales ||
            !fc2_scales)
            return fail(FP8G_ERR_INVALID_ARGUMENT, "null pointer argument");
        if (!aligned(input, 16) || !aligned(fc1_weights, 16) || !aligned(fc2_weights, 16) ||
            !aligned(out, 16) || !aligned(token_selected, 4) || !aligned(fc1_scales, 4) ||
            !aligned(fc2_scales, 4))
            return fail(FP8G_ERR_INVALID_ARGUMENT,
                        "input, weights and out must be 16-byte aligned, token_selected and "
                        "scales 4-byte aligned");
        const size_t need =
            moe_workspace(num_tokens, num_experts, top_k, hidden_size, inter_size).total;
        if (need > static_cast<size_t>(FP8G_MOE_STATIC_SCRATCH_BYTES))
            return fail(FP8G_ERR_UNSUPPORTED,
                        "this problem needs %zu bytes of scratch; the static scratch holds %zu "
                        "(use fused_moe_deepseek_fp8_block_scale with a workspace)",
                        need, static_cast<size_t>(FP8G_MOE_STATIC_SCRATCH_BYTES));
        DeviceState* ds = nullptr;
        if ((s = device_state(&ds)) != FP8G_OK) return s;
        uint8_t* scratch = nullptr;
        {
            std::lock_guard<std::mutex> lock(g_mutex);
            if (!ds->moe_static_scratch) {
                void* addr = nullptr;
                cudaError_t e = cudaGetSymbolAddress(&addr, g_moe_static_scratch);
                if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
                ds->moe_static_scratch = static_cast<uint8_t*>(addr);
            }
            scratch = ds->moe_static_scratch;
        }
        s = moe_run(*ds, input, token_selected, fc1_weights, fc2_weights, out, fc1_scales,
                    fc2_scales, num_tokens, num_experts, top_k, hidden_size, inter_size, scratch,
                    stream);
        if (s == FP8G_OK) t_last_error.clear();
        return s;
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

fp8g_status_t fused_moe_deepseek_fp8_block_scale_workspace_layout(
    int64_t num_tokens, int64_t num_experts, int64_t top_k, int64_t hidden_size,
    int64_t inter_size, int64_t* rows, size_t offsets[8]) {
    try {
        if (!rows || !offsets) return fail(FP8G_ERR_INVALID_ARGUMENT, "null pointer argument");
        fp8g_status_t s = check_moe_shape(num_tokens, num_experts, top_k, hidden_size,
                                          inter_size);
        if (s != FP8G_OK) return s;
        const MoeWorkspace w =
            moe_workspace(num_tokens, num_experts, top_k, hidden_size, inter_size);
        *rows = w.rows;
        const size_t at[8] = {w.m_indices, w.row_of, w.a1, w.a1_scale, w.h, w.a2, w.a2_scale, w.y};
        for (int i = 0; i < 8; ++i) offsets[i] = at[i];
        t_last_error.clear();
        return FP8G_OK;
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

fp8g_status_t fp8g_get_stream_status(unsigned int* flags, int clear, cudaStream_t stream) {
    try {
        if (!flags) return fail(FP8G_ERR_INVALID_ARGUMENT, "flags is null");
        DeviceState* ds = nullptr;
        fp8g_status_t s = device_state(&ds);
        if (s != FP8G_OK) return s;
        unsigned int v = 0;
        cudaError_t e = cudaMemcpyAsync(&v, ds->status, sizeof(v), cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess && clear) e = cudaMemsetAsync(ds->status, 0, sizeof(v), stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail(e, "reading the device status word on the stream");
        *flags = v;
        if (v & FP8G_DEVICE_TIMEOUT)
            return fail(FP8G_ERR_TIMEOUT, "a kernel gave up waiting on its pipeline (timeout)");
        t_last_error.clear();
        return FP8G_OK;
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

void fp8g_testing_set_wait_limit_ns(uint64_t ns) {
    t_wait_limit_ns = ns ? ns : fp8g::WAIT_LIMIT_NS;
}

int fp8g_testing_last_gemm_cta_pair(void) { return t_last_gemm_pair; }

fp8g_status_t fp8g_get_device_status(unsigned int* flags, int clear) {
    try {
        if (!flags) return fail(FP8G_ERR_INVALID_ARGUMENT, "flags is null");
        DeviceState* ds = nullptr;
        fp8g_status_t s = device_state(&ds);
        if (s != FP8G_OK) return s;
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        unsigned int v = 0;
        e = cudaMemcpy(&v, ds->status, sizeof(v), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
        if (clear) {
            e = cudaMemset(ds->status, 0, sizeof(unsigned int));
            if (e == cudaSuccess) e = cudaDeviceSynchronize();
            if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
        }
        *flags = v;
        if (v & FP8G_DEVICE_TIMEOUT)
            return fail(FP8G_ERR_TIMEOUT, "a kernel gave up waiting on its pipeline (timeout)");
        t_last_error.clear();
        return FP8G_OK;
    } catch (...) {
        return fail(FP8G_ERR_CUDA, "unexpected exception");
    }
}

}  // extern "C"
