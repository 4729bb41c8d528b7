// C-ABI entry points of libpa: argument checks, launch planning, launches.
// The operations and their sources are documented in include/pa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "pa.h"
#include "pa_decode.cuh"
#include "pa_decode_gqa.cuh"
#include "pa_decode_mha.cuh"
#include "pa_decode_q8.cuh"
#include "pa_decode_q8f.cuh"
#include "pa_decode_q8t.cuh"
#include "pa_internal.h"

namespace pa {

const void *reduce_kernel(int head_dim, bool wide) {
    if (head_dim == 64)
        return wide ? reinterpret_cast<const void *>(&pa_reduce_wide_kernel<64>)
                    : reinterpret_cast<const void *>(&pa_reduce_kernel<64>);
    if (head_dim == 128)
        return wide ? reinterpret_cast<const void *>(&pa_reduce_wide_kernel<128>)
                    : reinterpret_cast<const void *>(&pa_reduce_kernel<128>);
    return nullptr;
}

namespace {

thread_local std::string g_detail;

pa_status fail(pa_status st, const std::string &why) {
    g_detail = why;
    return st;
}

pa_status cuda_fail(cudaError_t e, const char *what) {
    g_detail = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return PA_ERR_CUDA;
}

int elt_bytes(int dtype) { return dtype == PA_F32 ? 4 : 2; }
bool dtype_ok(int dtype) { return dtype == PA_F32 || dtype == PA_F16 || dtype == PA_BF16; }
bool code_dtype_ok(int dtype) { return dtype == PA_I8 || dtype == PA_E4M3; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool block_size_ok(int bs) { return bs == 8 || bs == 16 || bs == 32; }
bool head_dim_ok(int d) { return d == 64 || d == 128; }

// Per-device facts and per-kernel launch settings, filled on first use.
std::mutex g_mu;
std::map<int, int> g_sms;
std::map<std::pair<int, const void *>, size_t> g_smem_set;
std::map<std::tuple<int, const void *, size_t>, int> g_occ;

cudaError_t device_sms(int *dev, int *sms) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sms.find(*dev);
    if (it != g_sms.end()) {
        *sms = it->second;
        return cudaSuccess;
    }
    e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev);
    if (e == cudaSuccess)
        g_sms[*dev] = *sms;
    return e;
}

cudaError_t prepare_kernel(int dev, const void *fn, size_t smem, int threads, int *blocks_per_sm) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(dev, fn);
    auto it = g_smem_set.find(key);
    if (it == g_smem_set.end() || it->second < smem) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
        g_smem_set[key] = smem;
    }
    auto okey = std::make_tuple(dev, fn, smem);
    auto oit = g_occ.find(okey);
    if (oit != g_occ.end()) {
        *blocks_per_sm = oit->second;
        return cudaSuccess;
    }
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, threads, smem);
    if (e != cudaSuccess)
        return e;
    g_occ[okey] = *blocks_per_sm;
    return cudaSuccess;
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link-time
// dependency on the driver library).
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn) {
    std::call_once(g_encode_once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
            g_encode_err = cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    *fn = g_encode;
    return g_encode_err;
}

// Encoded tensor maps, cached per thread: a map is a function of its base
// address, element type and shape alone, so a repeated call (the same cache,
// queries and shapes, as in a decode loop) reuses the encoding instead of
// calling cuTensorMapEncodeTiled again.  16 entries, least recently used out.
struct TmKey {
    int kind;
    const void *base;
    long long a, b, c, d, e;
    bool operator==(const TmKey &o) const {
        return kind == o.kind && base == o.base && a == o.a && b == o.b && c == o.c && d == o.d && e == o.e;
    }
};
struct TmCache {
    static constexpr int kEntries = 16;
    TmKey key[kEntries];
    CUtensorMap map[kEntries];
    unsigned use[kEntries];
    unsigned clock = 0;
    int n = 0;
};
thread_local TmCache t_tm;

bool tm_lookup(const TmKey &k, CUtensorMap *out) {
    for (int i = 0; i < t_tm.n; ++i) {
        if (t_tm.key[i] == k) {
            *out = t_tm.map[i];
            t_tm.use[i] = ++t_tm.clock;
            return true;
        }
    }
    return false;
}

void tm_store(const TmKey &k, const CUtensorMap &m) {
    int slot = t_tm.n;
    if (slot == TmCache::kEntries) {
        slot = 0;
        for (int i = 1; i < TmCache::kEntries; ++i)
            if (t_tm.use[i] < t_tm.use[slot])
                slot = i;
    } else {
        ++t_tm.n;
    }
    t_tm.key[slot] = k;
    t_tm.map[slot] = m;
    t_tm.use[slot] = ++t_tm.clock;
}

// 4-D view of a K or V cache [num_blocks * H_kv][block_size][head_dim] as
// [tile][128-byte segment of the row][row][elements of the segment]; one box is
// a whole (block, head) tile and lands in shared memory as one 128-byte-wide,
// block_size-row box per segment (128-byte swizzle).
pa_status kv_tensor_map(CUtensorMap *map, const void *base, int dtype, int head_dim, int block_size,
                        long long tiles) {
    const TmKey key{1, base, dtype, head_dim, block_size, tiles, 0};
    if (tm_lookup(key, map))
        return PA_OK;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = tensor_map_encoder(&enc);
    if (e != cudaSuccess || !enc)
        return cuda_fail(e == cudaSuccess ? cudaErrorSymbolNotFound : e, "cuTensorMapEncodeTiled lookup");
    const int elt = elt_bytes(dtype);
    const CUtensorMapDataType dt = dtype == PA_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t row = static_cast<cuuint64_t>(head_dim) * elt;
    const cuuint32_t segs = static_cast<cuuint32_t>(row / 128);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(128 / elt), static_cast<cuuint64_t>(block_size), segs,
                          static_cast<cuuint64_t>(tiles)};
    cuuint64_t strides[3] = {row, 128, row * block_size};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elt), static_cast<cuuint32_t>(block_size), segs, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, dt, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_INVALID_ARGUMENT, "cuTensorMapEncodeTiled rejected the cache layout (code " +
                                                 std::to_string(static_cast<int>(r)) + ")");
    tm_store(key, *map);
    return PA_OK;
}

// 5-D view of a 16-bit K or V cache with head_dim 128 for the tensor-core
// kernel: [tile = block * H_kv + head][row / 8][half][row % 8][64 elements];
// one box is `box_tiles` consecutive whole (block, head) tiles (1 for a paged
// cache; a contiguous cache's tiles of one kv head are consecutive) and lands
// in shared memory as 8-row groups of both 128-byte halves (128-byte swizzle).
pa_status kv_tensor_map_groups(CUtensorMap *map, const void *base, int dtype, int block_size, long long tiles,
                               int box_tiles = 1) {
    const TmKey key{2, base, dtype, block_size, tiles, box_tiles, 0};
    if (tm_lookup(key, map))
        return PA_OK;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = tensor_map_encoder(&enc);
    if (e != cudaSuccess || !enc)
        return cuda_fail(e == cudaSuccess ? cudaErrorSymbolNotFound : e, "cuTensorMapEncodeTiled lookup");
    const CUtensorMapDataType dt = dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t row = 256;  // bytes per token row (128 x 2 bytes)
    cuuint64_t dims[5] = {64, 8, 2, static_cast<cuuint64_t>(block_size / 8), static_cast<cuuint64_t>(tiles)};
    cuuint64_t strides[4] = {row, 128, 8 * row, row * block_size};
    cuuint32_t box[5] = {64, 8, 2, static_cast<cuuint32_t>(block_size / 8), static_cast<cuuint32_t>(box_tiles)};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, dt, 5, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_INVALID_ARGUMENT, "cuTensorMapEncodeTiled rejected the grouped cache view (code " +
                                                 std::to_string(static_cast<int>(r)) + ")");
    tm_store(key, *map);
    return PA_OK;
}

// 2-D view of q [num_seqs * num_heads][head_dim] with a box of one 128-byte
// row segment x `group` rows (the query heads of one kv head), 128-byte swizzle.
pa_status q_tensor_map(CUtensorMap *map, const void *base, int dtype, int head_dim, long long rows, int group) {
    const TmKey key{3, base, dtype, head_dim, rows, group, 0};
    if (tm_lookup(key, map))
        return PA_OK;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = tensor_map_encoder(&enc);
    if (e != cudaSuccess || !enc)
        return cuda_fail(e == cudaSuccess ? cudaErrorSymbolNotFound : e, "cuTensorMapEncodeTiled lookup");
    const int elt = elt_bytes(dtype);
    const CUtensorMapDataType dt = dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * elt};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elt), static_cast<cuuint32_t>(group)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_INVALID_ARGUMENT,
                    "cuTensorMapEncodeTiled rejected the query layout (code " + std::to_string(static_cast<int>(r)) + ")");
    tm_store(key, *map);
    return PA_OK;
}

// 3-D view of an 8-bit page pool [pages = block * H_kv + head][block_size +
// scale rows][128 bytes] for the tensor-core E4M3 kernel.  Codes: a box is the
// code rows of 4 adjacent pages (128-byte swizzle); scales: a box is the
// 4 * block_size scale bytes of the same 4 pages (no swizzle).
pa_status q8_page_tensor_map(CUtensorMap *map, const void *base, int block_size, long long pages, bool scales) {
    const TmKey key{4, base, block_size, pages, scales ? 1 : 0, 0, 0};
    if (tm_lookup(key, map))
        return PA_OK;
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = tensor_map_encoder(&enc);
    if (e != cudaSuccess || !enc)
        return cuda_fail(e == cudaSuccess ? cudaErrorSymbolNotFound : e, "cuTensorMapEncodeTiled lookup");
    const cuuint64_t rows = static_cast<cuuint64_t>(block_size + q8_scale_rows(block_size, 128));
    cuuint64_t dims[3] = {128, rows, static_cast<cuuint64_t>(pages)};
    cuuint64_t strides[2] = {128, rows * 128};
    cuuint32_t box[3] = {scales ? static_cast<cuuint32_t>(4 * block_size) : 128u,
                         scales ? 1u : static_cast<cuuint32_t>(block_size), static_cast<cuuint32_t>(kQ8tHeads)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, scales ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_INVALID_ARGUMENT, "cuTensorMapEncodeTiled rejected the 8-bit page layout (code " +
                                                 std::to_string(static_cast<int>(r)) + ")");
    tm_store(key, *map);
    return PA_OK;
}

constexpr int kDefaultPartition = 512;
// The tensor-core kernels (grouped heads over 16-bit K/V, and over E4M3
// pages) pay more per item (query load, the merge of the quarters, partials):
// their default partition is twice as long.  pa_decode_workspace_size(..., 0) sizes for the shorter one, which
// needs at least as much.
constexpr int kGqaDefaultPartition = 1024;
// The block size contiguous caches are cut into (their tiles: TMA boxes).
constexpr int kContiguousBlock = 16;
constexpr int kQ8fStageBudget = 48 * 1024;
// Grouped heads: 3 stages of 4 kv heads' pages at block 16 (17.4 KB each; 3 CTAs
// per SM still fit).  Measured on the GQA INT8 batch: 2 stages 0.200 ms, 3
// stages 0.197 ms, 4 stages 0.226 ms (2 CTAs per SM).
constexpr int kQ8fGroupStageBudget = 56 * 1024;
constexpr int kMhaStageBudget = 64 * 1024;
constexpr int kGqaStages = 3;
constexpr int kStageBudget = 48 * 1024;

// Whether pa_decode of this shape takes the tensor-core grouped-head kernel
// (16-bit K/V, head_dim 128, query groups of 2, 4 or 8; the pool and batch
// size limits of launch_decode_kernel aside).
bool gqa_tensor_core_path(int num_heads, int num_kv_heads, int head_dim, int dtype) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return false;
    const int G = num_heads / num_kv_heads;
    return (G == 2 || G == 4 || G == 8) && head_dim == 128 && (dtype == PA_F16 || dtype == PA_BF16);
}

// Whether pa_decode_quant of this shape takes the tensor-core E4M3 kernel
// (the pool and batch size limits of launch_decode_q8_kernel aside).
bool q8t_tensor_core_path(int num_heads, int num_kv_heads, int head_dim, int block_size, int q_dtype,
                          int cache_dtype) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return false;
    const int G = num_heads / num_kv_heads;
    return cache_dtype == PA_E4M3 && head_dim == 128 && G >= 2 && G <= kQ8tMaxG &&
           (block_size == 16 || block_size == 32) && num_kv_heads % kQ8tHeads == 0 &&
           (q_dtype == PA_F16 || q_dtype == PA_BF16);
}

struct DecodePlan {
    int bpp = 0;
    int max_parts = 0;
    size_t workspace = 0;
};

pa_status plan_decode(int num_seqs, int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                      int window, int partition_size, DecodePlan *plan) {
    if (num_seqs < 0 || num_heads <= 0 || max_blocks_per_seq <= 0 || window < 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_seqs, num_heads, max_blocks_per_seq or window out of range");
    if (!block_size_ok(block_size))
        return fail(PA_ERR_UNSUPPORTED, "block_size must be 8, 16 or 32");
    if (!head_dim_ok(head_dim))
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    int P = partition_size == 0 ? kDefaultPartition : partition_size;
    if (P <= 0 || P % block_size != 0 || P / block_size > kMaxBpp)
        return fail(PA_ERR_INVALID_ARGUMENT, "partition_size must be a positive multiple of block_size, at most 256 blocks");
    plan->bpp = P / block_size;
    long long span_blocks = max_blocks_per_seq;
    if (window > 0) {
        const long long wb = (static_cast<long long>(window) + block_size - 1) / block_size + 1;
        if (wb < span_blocks)
            span_blocks = wb;
    }
    plan->max_parts = static_cast<int>((span_blocks + plan->bpp - 1) / plan->bpp);
    if (plan->max_parts > 1)
        plan->workspace = static_cast<size_t>(num_seqs) * num_heads * plan->max_parts * (head_dim + 2) * sizeof(float);
    else
        plan->workspace = 0;
    return PA_OK;
}

}  // namespace

void set_last_error_detail(const char *why) { g_detail = why; }

// Item counters for the kernels that claim their items (DecodeParams::work):
// zero when the module loads, and every launch returns its pair to zero.
// Eager launches take pairs round-robin from the first kWorkSlots, so
// launches in flight at the same time (up to kWorkSlots of them) never share
// one.  A launch captured into a CUDA graph keeps its pair for every replay,
// so it takes one of the next kCapturedSlots pairs for good: no eager launch
// and no other captured launch ever gets it.  Once those are spent, captured
// launches run without a counter (each CTA takes a fixed stride of items:
// the same results, less even balance).
constexpr int kWorkSlots = 4096;
constexpr int kCapturedSlots = 4096;
constexpr int kMaxDevices = 64;
__device__ unsigned int g_work[2 * (kWorkSlots + kCapturedSlots)];

unsigned int *work_counter(int device, cudaStream_t stream) {
    static unsigned int *base[kMaxDevices] = {};
    static std::mutex mu;
    static std::atomic<unsigned int> next{0};
    static std::atomic<int> next_captured[kMaxDevices] = {};
    if (device < 0 || device >= kMaxDevices)
        return nullptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;  // status unknown: no counter
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!base[device]) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_work) != cudaSuccess)
                return nullptr;
            base[device] = static_cast<unsigned int *>(ptr);
        }
    }
    if (cap != cudaStreamCaptureStatusNone) {
        const int k = next_captured[device].fetch_add(1);
        return k < kCapturedSlots ? base[device] + 2 * (kWorkSlots + k) : nullptr;
    }
    return base[device] + 2 * (next.fetch_add(1u) % kWorkSlots);
}

// The partition reduce: a warp per row when there are rows enough to fill the
// GPU and few partitions each, else a CTA per row.
static cudaError_t launch_reduce(DecodeParams &p, int head_dim, long long rows, cudaStream_t cs) {
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return e;
    const bool wide = rows < 8LL * sms || p.max_parts > 32;
    void *args[] = {&p};
    const long long grid = wide ? rows : (rows + kReduceRows - 1) / kReduceRows;
    return launch_dependent(reduce_kernel(head_dim, wide), dim3(static_cast<unsigned>(grid)),
                            dim3(wide ? kReduceWideThreads : kReduceThreads), args, 0, cs);
}

pa_status launch_decode_kernel(DecodeParams &p, int dtype, int head_dim, int G, cudaStream_t cs) {
    const int block_size = p.block_size;
    const int row = head_dim * elt_bytes(dtype);
    const int tile = block_size * row;
    // a paged pool holds num_blocks x H_kv tiles; a contiguous cache
    // num_seqs x H_kv x max_blocks_per_seq
    const long long tiles = p.contiguous
                                ? static_cast<long long>(p.num_seqs) * p.num_kv_heads * p.max_blocks_per_seq
                                : static_cast<long long>(p.num_blocks) * p.num_kv_heads;
    // MHA takes the TMA-tensor kernel; its 3-D tensor map addresses tiles with
    // a 32-bit coordinate, so very large pools use the general kernel.
    const bool mha = (G == 1 && tiles <= INT_MAX);
    // Grouped heads with 16-bit K/V and head_dim 128 take the tensor-core kernel.
    const bool gqa_tc = (G > 1 && head_dim == 128 && dtype != PA_F32 && tiles <= INT_MAX &&
                         static_cast<long long>(p.num_seqs) * p.num_heads <= INT_MAX);
    const void *fn;
    size_t smem;
    int threads;
    CUtensorMap tmk, tmv, tmq, tmkw, tmvw;
    if (p.contiguous && !gqa_tc && !mha)
        return fail(PA_ERR_UNSUPPORTED, "contiguous caches take one query head per kv head, or 2, 4 or 8 with "
                                        "fp16 / bf16 K/V and head_dim 128");
    if (gqa_tc) {
        fn = dtype == PA_F16 ? decode_gqa_kernel_f16(block_size, G) : decode_gqa_kernel_bf16(block_size, G);
        p.stages = kGqaStages;
        smem = gqa_smem_layout(kGqaStages).total;
        threads = kGqaThreads;
        pa_status ts = kv_tensor_map_groups(&tmk, p.k_cache, dtype, block_size, tiles);
        if (ts == PA_OK)
            ts = kv_tensor_map_groups(&tmv, p.v_cache, dtype, block_size, tiles);
        if (ts == PA_OK)
            ts = q_tensor_map(&tmq, p.q, dtype, head_dim, static_cast<long long>(p.num_seqs) * p.num_heads, G);
        tmkw = tmk;
        tmvw = tmv;
        if (ts == PA_OK && p.contiguous) {
            // a whole 128-token tile of a contiguous cache in one copy
            ts = kv_tensor_map_groups(&tmkw, p.k_cache, dtype, block_size, tiles, kTileTokens / block_size);
            if (ts == PA_OK)
                ts = kv_tensor_map_groups(&tmvw, p.v_cache, dtype, block_size, tiles, kTileTokens / block_size);
        }
        if (ts != PA_OK)
            return ts;
    } else if (mha) {
        fn = dtype == PA_F32   ? decode_mha_kernel_f32(head_dim, block_size)
             : dtype == PA_F16 ? decode_mha_kernel_f16(head_dim, block_size)
                               : decode_mha_kernel_bf16(head_dim, block_size);
        // the stages form one sub-ring per consumer warp: a multiple of their count
        int S = kMhaStageBudget / (2 * tile);
        S -= S % kMhaWarps;
        S = S < kMhaWarps ? kMhaWarps : (S > 16 ? 16 : S);
        p.stages = S;
        smem = mha_smem_layout(S, tile, row, head_dim).total;
        threads = kMhaThreads;
        pa_status ts = kv_tensor_map(&tmk, p.k_cache, dtype, head_dim, block_size, tiles);
        if (ts == PA_OK)
            ts = kv_tensor_map(&tmv, p.v_cache, dtype, head_dim, block_size, tiles);
        if (ts != PA_OK)
            return ts;
    } else {
        fn = dtype == PA_F32   ? decode_kernel_f32(head_dim, G)
             : dtype == PA_F16 ? decode_kernel_f16(head_dim, G)
                               : decode_kernel_bf16(head_dim, G);
        int S = kStageBudget / (2 * tile);
        S = S < 2 ? 2 : (S > 8 ? 8 : S);
        p.stages = S;
        smem = decode_smem_layout(S, tile, row, G, head_dim).total;
        threads = kDecodeThreads;
    }
    if (!fn)
        return fail(PA_ERR_UNSUPPORTED, "no decode kernel for this dtype / head_dim / group / block size");

    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    e = prepare_kernel(dev, fn, smem, threads, &per_sm);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode kernel set-up");
    if (per_sm < 1)
        return fail(PA_ERR_UNSUPPORTED, "decode kernel does not fit on an SM");

    const long long items_max = static_cast<long long>(p.num_seqs) * p.num_kv_heads * p.max_parts;
    long long grid = static_cast<long long>(sms) * per_sm;
    if (grid > items_max)
        grid = items_max;
    if (grid < 1)
        grid = 1;
    // the TMA-fed kernels claim their items from a per-launch counter
    // (balances contexts of mixed lengths) when there are more items than
    // CTAs; with a CTA for every item, each takes its own (no atomic on the
    // path of a small, latency-bound launch)
    if ((gqa_tc || mha) && items_max > grid)
        p.work = work_counter(dev, cs);
    void *args_gqa[] = {&p, &tmk, &tmv, &tmq, &tmkw, &tmvw};
    void *args_mha[] = {&p, &tmk, &tmv};
    void *args[] = {&p};
    e = launch_dependent(fn, dim3(static_cast<unsigned>(grid)), dim3(threads),
                         gqa_tc ? args_gqa : (mha ? args_mha : args), smem, cs);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode launch");
    return PA_OK;
}

pa_status launch_decode_q8_kernel(DecodeParams &p, int cache_dtype, int head_dim, int G, cudaStream_t cs) {
    const long long tiles = static_cast<long long>(p.num_blocks) * p.num_kv_heads;
    // E4M3 pages, grouped heads, head_dim 128, block size 16 / 32, kv heads in
    // fours, 16-bit queries: the tensor-core kernel (kind::f8f6f4 on the codes).
    // One query per kv head stays on the TMA-fed CUDA-core kernel, which is
    // faster there.
    const bool tc = cache_dtype == PA_E4M3 && head_dim == 128 && G >= 2 && G <= kQ8tMaxG &&
                    (p.block_size == 16 || p.block_size == 32) && p.num_kv_heads % kQ8tHeads == 0 &&
                    (p.q_dtype == PA_F16 || p.q_dtype == PA_BF16) && tiles <= INT_MAX &&
                    static_cast<long long>(p.num_seqs) * p.num_heads <= INT_MAX;
    if (tc) {
        const void *tfn = decode_q8t_kernel_e4m3(G, p.block_size);
        if (!tfn)
            return fail(PA_ERR_UNSUPPORTED, "no tensor-core E4M3 decode kernel for this group / block size");
        CUtensorMap tmk, tmv, tsk, tsv;
        pa_status ts = q8_page_tensor_map(&tmk, p.k_cache, p.block_size, tiles, false);
        if (ts == PA_OK)
            ts = q8_page_tensor_map(&tmv, p.v_cache, p.block_size, tiles, false);
        if (ts == PA_OK)
            ts = q8_page_tensor_map(&tsk, p.k_cache, p.block_size, tiles, true);
        if (ts == PA_OK)
            ts = q8_page_tensor_map(&tsv, p.v_cache, p.block_size, tiles, true);
        if (ts != PA_OK)
            return ts;
        p.stages = kQ8tStages;
        const size_t smem = q8t_smem_layout(kQ8tStages).total;
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = device_sms(&dev, &sms);
        if (e != cudaSuccess)
            return cuda_fail(e, "device query");
        e = prepare_kernel(dev, tfn, smem, kQ8tThreads, &per_sm);
        if (e != cudaSuccess)
            return cuda_fail(e, "decode kernel set-up");
        if (per_sm < 1)
            return fail(PA_ERR_UNSUPPORTED, "decode kernel does not fit on an SM");
        const long long items_max =
            static_cast<long long>(p.num_seqs) * (p.num_kv_heads / kQ8tHeads) * p.max_parts;
        // one CTA per SM: each holds all of an SM's tensor memory
        long long grid = sms;
        if (grid > items_max)
            grid = items_max;
        if (grid < 1)
            grid = 1;
        // items are claimed from a per-launch counter (balances contexts of
        // mixed lengths) when there are more items than CTAs; otherwise each
        // CTA takes its own
        if (items_max > grid)
            p.work = work_counter(dev, cs);
        void *args[] = {&p, &tmk, &tmv, &tsk, &tsv};
        e = launch_dependent(tfn, dim3(static_cast<unsigned>(grid)), dim3(kQ8tThreads), args, smem, cs);
        if (e != cudaSuccess)
            return cuda_fail(e, "decode launch");
        return PA_OK;
    }
    // head_dim 128, up to 4 query heads per kv head: the TMA-fed kernel (E4M3
    // multiplies fp16 queries, so fp32 queries stay on the general kernel)
    const bool fast = head_dim == 128 && G <= 4 && tiles <= INT_MAX &&
                      !(cache_dtype == PA_E4M3 && p.q_dtype == PA_F32);
    if (fast) {
        const void *ffn = cache_dtype == PA_I8 ? decode_q8f_kernel_i8(G, p.block_size)
                                               : decode_q8f_kernel_e4m3(G, p.block_size);
        if (!ffn)
            return fail(PA_ERR_UNSUPPORTED, "no 8-bit-cache decode kernel for this group / block size");
        // a stage holds the K and V pages of 4 kv heads; every consumer warp
        // reads every stage
        const int stage = 2 * kQ8fWarps * q8_page_bytes(p.block_size, kQ8fD);
        int S = (G > 1 ? kQ8fGroupStageBudget : kQ8fStageBudget) / stage;
        S = S < 2 ? 2 : (S > 8 ? 8 : S);
        p.stages = S;
        const size_t smem = q8f_smem_layout(S, p.block_size, G, kQ8fD * (p.q_dtype == PA_F32 ? 4 : 2)).total;
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = device_sms(&dev, &sms);
        if (e != cudaSuccess)
            return cuda_fail(e, "device query");
        e = prepare_kernel(dev, ffn, smem, kQ8fThreads, &per_sm);
        if (e != cudaSuccess)
            return cuda_fail(e, "decode kernel set-up");
        if (per_sm < 1)
            return fail(PA_ERR_UNSUPPORTED, "decode kernel does not fit on an SM");
        const long long items_max = static_cast<long long>(p.num_seqs) *
                                    ((p.num_kv_heads + kQ8fWarps - 1) / kQ8fWarps) * p.max_parts;
        long long grid = static_cast<long long>(sms) * per_sm;
        if (grid > items_max)
            grid = items_max;
        if (grid < 1)
            grid = 1;
        if (items_max > grid)
            p.work = work_counter(dev, cs);  // items claimed from a per-launch counter
        void *args[] = {&p};
        e = launch_dependent(ffn, dim3(static_cast<unsigned>(grid)), dim3(kQ8fThreads), args, smem, cs);
        if (e != cudaSuccess)
            return cuda_fail(e, "decode launch");
        return PA_OK;
    }
    const void *fn = cache_dtype == PA_I8 ? decode_q8_kernel_i8(head_dim, G) : decode_q8_kernel_e4m3(head_dim, G);
    if (!fn)
        return fail(PA_ERR_UNSUPPORTED, "no 8-bit-cache decode kernel for this head_dim / group");
    const int stage = static_cast<int>(q8_stage_bytes(p.block_size, head_dim));
    int S = kStageBudget / stage;
    S = S < 2 ? 2 : (S > 16 ? 16 : S);
    p.stages = S;
    const size_t smem = q8_smem_layout(S, p.block_size, G, head_dim).total;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    e = prepare_kernel(dev, fn, smem, kDecodeThreads, &per_sm);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode kernel set-up");
    if (per_sm < 1)
        return fail(PA_ERR_UNSUPPORTED, "decode kernel does not fit on an SM");
    const long long items_max = static_cast<long long>(p.num_seqs) * p.num_kv_heads * p.max_parts;
    long long grid = static_cast<long long>(sms) * per_sm;
    if (grid > items_max)
        grid = items_max;
    if (grid < 1)
        grid = 1;
    void *args[] = {&p};
    e = launch_dependent(fn, dim3(static_cast<unsigned>(grid)), dim3(kDecodeThreads), args, smem, cs);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode launch");
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                                int window, int partition_size) {
    DecodePlan plan;
    if (plan_decode(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq, window, partition_size, &plan) !=
        PA_OK)
        return 0;
    return plan.workspace;
}

pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
                    const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, float scale, int window, pa_dtype dtype, pa_dtype out_dtype,
                    int max_blocks_per_seq, int num_blocks, int partition_size, void *workspace,
                    size_t workspace_bytes, uint32_t *err_word, pa_stream_t stream) {
    g_detail.clear();
    if (partition_size == 0 && gqa_tensor_core_path(num_heads, num_kv_heads, head_dim, dtype))
        partition_size = kGqaDefaultPartition;
    DecodePlan plan;
    pa_status st = plan_decode(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq, window,
                               partition_size, &plan);
    if (st != PA_OK)
        return st;
    if (num_seqs == 0)
        return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_heads must be a multiple of num_kv_heads");
    const int G = num_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PA_ERR_UNSUPPORTED, "num_heads / num_kv_heads must be 1, 2, 4 or 8");
    if (!dtype_ok(dtype) || !dtype_ok(out_dtype))
        return fail(PA_ERR_INVALID_ARGUMENT, "unknown dtype");
    if (num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_blocks must be positive");
    if (!std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARGUMENT, "scale must be finite");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARGUMENT, "q, k_cache and v_cache must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(out) & (elt_bytes(out_dtype) - 1)) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "out is not aligned to its element size");
    if (plan.workspace > 0 && (workspace == nullptr || workspace_bytes < plan.workspace))
        return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace smaller than pa_decode_workspace_size()");
    if (plan.workspace > 0 && !aligned16(workspace))
        return fail(PA_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");

    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    const size_t acc_floats = static_cast<size_t>(num_seqs) * num_heads * plan.max_parts * head_dim;
    p.part_acc = plan.workspace ? static_cast<float *>(workspace) : nullptr;
    p.part_ml = plan.workspace ? static_cast<float *>(workspace) + acc_floats : nullptr;
    p.err = err_word;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = block_size;
    p.window = window;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_len = static_cast<int>(std::min<long long>(static_cast<long long>(max_blocks_per_seq) * block_size, INT_MAX));
    p.num_blocks = num_blocks;
    p.bpp = plan.bpp;
    p.max_parts = plan.max_parts;
    p.out_dtype = out_dtype;
    p.stages = 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.start_tok = nullptr;
    p.force_partial = 0;
    p.q_dtype = dtype;

    const pa_status ls = launch_decode_kernel(p, dtype, head_dim, G, reinterpret_cast<cudaStream_t>(stream));
    if (ls != PA_OK)
        return ls;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (plan.max_parts > 1) {
        const long long rows = static_cast<long long>(num_seqs) * num_heads;
        const cudaError_t e = launch_reduce(p, head_dim, rows, cs);
        if (e != cudaSuccess)
            return cuda_fail(e, "reduce launch");
    }
    return PA_OK;
}

pa_status pa_append_kv(const void *k, const void *v, const int64_t *slot_mapping, void *k_cache, void *v_cache,
                       int num_tokens, int num_kv_heads, int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                       uint32_t *err_word, pa_stream_t stream) {
    g_detail.clear();
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_tokens, num_kv_heads or num_blocks out of range");
    if (!block_size_ok(block_size))
        return fail(PA_ERR_UNSUPPORTED, "block_size must be 8, 16 or 32");
    if (!head_dim_ok(head_dim))
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (!dtype_ok(dtype))
        return fail(PA_ERR_INVALID_ARGUMENT, "unknown dtype");
    if (num_tokens == 0)
        return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARGUMENT, "k, v and the caches must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "slot_mapping must be 8-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    e = launch_append(k, v, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads, head_dim * elt_bytes(dtype),
                      block_size, num_blocks, err_word, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "append launch");
    return PA_OK;
}

pa_status pa_copy_blocks(const int64_t *src_dst_pairs, int num_pairs, void *k_cache, void *v_cache, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype, uint32_t *err_word,
                         pa_stream_t stream) {
    g_detail.clear();
    if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_pairs, num_kv_heads or num_blocks out of range");
    if (!block_size_ok(block_size))
        return fail(PA_ERR_UNSUPPORTED, "block_size must be 8, 16 or 32");
    if (!head_dim_ok(head_dim))
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (!dtype_ok(dtype))
        return fail(PA_ERR_INVALID_ARGUMENT, "unknown dtype");
    if (num_pairs == 0)
        return PA_OK;
    if (!src_dst_pairs || !k_cache || !v_cache)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARGUMENT, "the caches must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "src_dst_pairs must be 8-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    const long long block_bytes =
        static_cast<long long>(num_kv_heads) * block_size * head_dim * elt_bytes(dtype);
    e = launch_copy_blocks(src_dst_pairs, num_pairs, k_cache, v_cache, block_bytes, num_blocks, err_word, sms,
                           reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "copy_blocks launch");
    return PA_OK;
}

pa_status pa_swap_blocks(const int64_t *src_dst_pairs, int num_pairs, const void *src_k, const void *src_v,
                         void *dst_k, void *dst_v, int src_num_blocks, int dst_num_blocks, int num_kv_heads,
                         int head_dim, int block_size, pa_dtype dtype, uint32_t *err_word, pa_stream_t stream) {
    g_detail.clear();
    if (num_pairs < 0 || num_kv_heads <= 0 || src_num_blocks <= 0 || dst_num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_pairs, num_kv_heads or a pool size out of range");
    if (!block_size_ok(block_size))
        return fail(PA_ERR_UNSUPPORTED, "block_size must be 8, 16 or 32");
    if (!head_dim_ok(head_dim))
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (!dtype_ok(dtype))
        return fail(PA_ERR_INVALID_ARGUMENT, "unknown dtype");
    if (num_pairs == 0)
        return PA_OK;
    if (!src_dst_pairs || !src_k || !src_v || !dst_k || !dst_v)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
        return fail(PA_ERR_INVALID_ARGUMENT, "the pools must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "src_dst_pairs must be 8-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    const long long block_bytes =
        static_cast<long long>(num_kv_heads) * block_size * head_dim * elt_bytes(dtype);
    e = launch_swap_blocks(src_dst_pairs, num_pairs, src_k, src_v, dst_k, dst_v, block_bytes, src_num_blocks,
                           dst_num_blocks, err_word, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "swap_blocks launch");
    return PA_OK;
}

size_t pa_quant_page_bytes(int head_dim, int block_size) {
    if (!head_dim_ok(head_dim) || !block_size_ok(block_size))
        return 0;
    return static_cast<size_t>(q8_page_bytes(block_size, head_dim));
}

pa_status pa_decode_contiguous(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                               int head_dim, int max_context_len, float scale, int window, pa_dtype dtype,
                               pa_dtype out_dtype, int partition_size, void *workspace, size_t workspace_bytes,
                               uint32_t *err_word, pa_stream_t stream) {
    g_detail.clear();
    constexpr int kBs = kContiguousBlock;
    if (max_context_len <= 0 || max_context_len % kBs != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "max_context_len must be a positive multiple of 16");
    const int mb = max_context_len / kBs;
    if (partition_size == 0 && gqa_tensor_core_path(num_heads, num_kv_heads, head_dim, dtype))
        partition_size = kGqaDefaultPartition;
    DecodePlan plan;
    pa_status st = plan_decode(num_seqs, num_heads, head_dim, kBs, mb, window, partition_size, &plan);
    if (st != PA_OK)
        return st;
    if (num_seqs == 0)
        return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !context_lens)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_heads must be a multiple of num_kv_heads");
    const int G = num_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PA_ERR_UNSUPPORTED, "num_heads / num_kv_heads must be 1, 2, 4 or 8");
    if (!dtype_ok(dtype) || !dtype_ok(out_dtype))
        return fail(PA_ERR_INVALID_ARGUMENT, "unknown dtype");
    if (G > 1 && !gqa_tensor_core_path(num_heads, num_kv_heads, head_dim, dtype))
        return fail(PA_ERR_UNSUPPORTED, "contiguous caches with grouped heads take fp16 / bf16 K/V and head_dim 128");
    if (!std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARGUMENT, "scale must be finite");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARGUMENT, "q, k_cache and v_cache must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(out) & (elt_bytes(out_dtype) - 1)) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "out is not aligned to its element size");
    if (static_cast<long long>(num_seqs) * num_kv_heads * mb > INT_MAX)
        return fail(PA_ERR_UNSUPPORTED, "contiguous cache too large for 32-bit tile indices");
    if (plan.workspace > 0 && (workspace == nullptr || workspace_bytes < plan.workspace))
        return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace smaller than pa_decode_workspace_size()");
    if (plan.workspace > 0 && !aligned16(workspace))
        return fail(PA_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");

    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = nullptr;  // never read: block b of a sequence is its b-th tile
    p.context_lens = context_lens;
    const size_t acc_floats = static_cast<size_t>(num_seqs) * num_heads * plan.max_parts * head_dim;
    p.part_acc = plan.workspace ? static_cast<float *>(workspace) : nullptr;
    p.part_ml = plan.workspace ? static_cast<float *>(workspace) + acc_floats : nullptr;
    p.err = err_word;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = kBs;
    p.window = window;
    p.max_blocks_per_seq = mb;
    p.max_len = max_context_len;
    p.num_blocks = mb;  // logical block ids stand in for table entries
    p.bpp = plan.bpp;
    p.max_parts = plan.max_parts;
    p.out_dtype = out_dtype;
    p.stages = 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.start_tok = nullptr;
    p.force_partial = 0;
    p.q_dtype = dtype;
    p.contiguous = 1;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const pa_status ls = launch_decode_kernel(p, dtype, head_dim, G, cs);
    if (ls != PA_OK)
        return ls;
    if (plan.max_parts > 1) {
        const cudaError_t e = launch_reduce(p, head_dim, static_cast<long long>(num_seqs) * num_heads, cs);
        if (e != cudaSuccess)
            return cuda_fail(e, "reduce launch");
    }
    return PA_OK;
}

pa_status pa_decode_quant(void *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens,
                          int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                          int window, pa_dtype dtype, pa_dtype cache_dtype, pa_dtype out_dtype,
                          int max_blocks_per_seq, int num_blocks, int partition_size, void *workspace,
                          size_t workspace_bytes, uint32_t *err_word, pa_stream_t stream) {
    g_detail.clear();
    if (partition_size == 0 &&
        q8t_tensor_core_path(num_heads, num_kv_heads, head_dim, block_size, dtype, cache_dtype))
        partition_size = kGqaDefaultPartition;
    DecodePlan plan;
    pa_status st = plan_decode(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq, window,
                               partition_size, &plan);
    if (st != PA_OK)
        return st;
    if (num_seqs == 0)
        return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_heads must be a multiple of num_kv_heads");
    const int G = num_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(PA_ERR_UNSUPPORTED, "num_heads / num_kv_heads must be 1, 2, 4 or 8");
    if (!dtype_ok(dtype) || !dtype_ok(out_dtype) || !code_dtype_ok(cache_dtype))
        return fail(PA_ERR_INVALID_ARGUMENT, "unknown dtype (q and out: PA_F32/F16/BF16; cache: PA_I8/PA_E4M3)");
    if (num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_blocks must be positive");
    if (!std::isfinite(scale))
        return fail(PA_ERR_INVALID_ARGUMENT, "scale must be finite");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARGUMENT, "q and the page pools must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(out) & (elt_bytes(out_dtype) - 1)) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "out is not aligned to its element size");
    if (plan.workspace > 0 && (workspace == nullptr || workspace_bytes < plan.workspace))
        return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace smaller than pa_decode_workspace_size()");
    if (plan.workspace > 0 && !aligned16(workspace))
        return fail(PA_ERR_INVALID_ARGUMENT, "workspace must be 16-byte aligned");

    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    const size_t acc_floats = static_cast<size_t>(num_seqs) * num_heads * plan.max_parts * head_dim;
    p.part_acc = plan.workspace ? static_cast<float *>(workspace) : nullptr;
    p.part_ml = plan.workspace ? static_cast<float *>(workspace) + acc_floats : nullptr;
    p.err = err_word;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = block_size;
    p.window = window;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_len = static_cast<int>(std::min<long long>(static_cast<long long>(max_blocks_per_seq) * block_size, INT_MAX));
    p.num_blocks = num_blocks;
    p.bpp = plan.bpp;
    p.max_parts = plan.max_parts;
    p.out_dtype = out_dtype;
    p.stages = 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.start_tok = nullptr;
    p.force_partial = 0;
    p.q_dtype = dtype;

    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const pa_status ls = launch_decode_q8_kernel(p, cache_dtype, head_dim, G, cs);
    if (ls != PA_OK)
        return ls;
    if (plan.max_parts > 1) {
        const long long rows = static_cast<long long>(num_seqs) * num_heads;
        cudaError_t e = launch_reduce(p, head_dim, rows, cs);
        if (e != cudaSuccess)
            return cuda_fail(e, "reduce launch");
    }
    return PA_OK;
}

pa_status pa_append_kv_quant(const void *k, const void *v, const int64_t *slot_mapping, void *k_cache, void *v_cache,
                             int num_tokens, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                             pa_dtype dtype, pa_dtype cache_dtype, uint32_t *err_word, pa_stream_t stream) {
    g_detail.clear();
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_tokens, num_kv_heads or num_blocks out of range");
    if (!block_size_ok(block_size))
        return fail(PA_ERR_UNSUPPORTED, "block_size must be 8, 16 or 32");
    if (!head_dim_ok(head_dim))
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (!dtype_ok(dtype) || !code_dtype_ok(cache_dtype))
        return fail(PA_ERR_INVALID_ARGUMENT, "unknown dtype (rows: PA_F32/F16/BF16; cache: PA_I8/PA_E4M3)");
    if (num_tokens == 0)
        return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARGUMENT, "k, v and the page pools must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "slot_mapping must be 8-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    e = launch_append_quant(k, v, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads, head_dim, dtype,
                            cache_dtype, block_size, num_blocks, err_word, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "append launch");
    return PA_OK;
}

pa_status pa_copy_blocks_quant(const int64_t *src_dst_pairs, int num_pairs, void *k_cache, void *v_cache,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks, uint32_t *err_word,
                               pa_stream_t stream) {
    g_detail.clear();
    if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_pairs, num_kv_heads or num_blocks out of range");
    if (!block_size_ok(block_size))
        return fail(PA_ERR_UNSUPPORTED, "block_size must be 8, 16 or 32");
    if (!head_dim_ok(head_dim))
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (num_pairs == 0)
        return PA_OK;
    if (!src_dst_pairs || !k_cache || !v_cache)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARGUMENT, "the page pools must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "src_dst_pairs must be 8-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    const long long block_bytes = static_cast<long long>(num_kv_heads) * q8_page_bytes(block_size, head_dim);
    e = launch_copy_blocks(src_dst_pairs, num_pairs, k_cache, v_cache, block_bytes, num_blocks, err_word, sms,
                           reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "copy_blocks launch");
    return PA_OK;
}

pa_status pa_swap_blocks_quant(const int64_t *src_dst_pairs, int num_pairs, const void *src_k, const void *src_v,
                               void *dst_k, void *dst_v, int src_num_blocks, int dst_num_blocks, int num_kv_heads,
                               int head_dim, int block_size, uint32_t *err_word, pa_stream_t stream) {
    g_detail.clear();
    if (num_pairs < 0 || num_kv_heads <= 0 || src_num_blocks <= 0 || dst_num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "num_pairs, num_kv_heads or a pool size out of range");
    if (!block_size_ok(block_size))
        return fail(PA_ERR_UNSUPPORTED, "block_size must be 8, 16 or 32");
    if (!head_dim_ok(head_dim))
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (num_pairs == 0)
        return PA_OK;
    if (!src_dst_pairs || !src_k || !src_v || !dst_k || !dst_v)
        return fail(PA_ERR_INVALID_ARGUMENT, "null pointer");
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
        return fail(PA_ERR_INVALID_ARGUMENT, "the pools must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u) != 0)
        return fail(PA_ERR_INVALID_ARGUMENT, "src_dst_pairs must be 8-byte aligned");
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    const long long block_bytes = static_cast<long long>(num_kv_heads) * q8_page_bytes(block_size, head_dim);
    e = launch_swap_blocks(src_dst_pairs, num_pairs, src_k, src_v, dst_k, dst_v, block_bytes, src_num_blocks,
                           dst_num_blocks, err_word, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "swap_blocks launch");
    return PA_OK;
}

const char *pa_status_string(pa_status status) {
    switch (status) {
    case PA_OK:
        return "PA_OK";
    case PA_ERR_INVALID_ARGUMENT:
        return "PA_ERR_INVALID_ARGUMENT";
    case PA_ERR_UNSUPPORTED:
        return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE_TOO_SMALL:
        return "PA_ERR_WORKSPACE_TOO_SMALL";
    case PA_ERR_CUDA:
        return "PA_ERR_CUDA";
    case PA_ERR_NO_BLOCKS:
        return "PA_ERR_NO_BLOCKS";
    }
    return "PA_ERR_UNKNOWN";
}

const char *pa_last_error_detail(void) { return g_detail.c_str(); }

int pa_version(void) { return (0 << 16) | (1 << 8) | 0; }

}  // extern "C"
