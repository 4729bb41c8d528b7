// KV append and copy-on-write block copy.
//
// Append ("PagedAttention — 把 KV cache 当虚拟内存页来管理", 核心要点: every
// generated token's key/value is saved; 案例 2: slot = physical block *
// block_size + offset): token i's rows go to
//   cache[slot / block_size][h][slot % block_size][:].
// Block copy (same page, 案例 3: copy-on-write, one whole block is the copy
// unit): for each (src, dst) pair the block's tiles of every kv head, K and V.
// Swap (same page, 踩过的坑: swap is the fallback when memory runs short): the
// block copy between two pools, one of which may be host memory.
// All are bit-exact 16-byte vector copies; bad slots / pairs are skipped and
// flagged in the error word.
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_quant.cuh"

namespace pa {

namespace {

__device__ inline uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// One thread moves one 16-byte chunk of a K row and the matching V chunk.
// Work index order: token, kv head, chunk -> reads of k / v are contiguous
// and each (token, head) row is written as one contiguous run.
__global__ void __launch_bounds__(256) append_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                     const int64_t *__restrict__ slots, uint4 *k_cache,
                                                     uint4 *v_cache, long long num_tokens, int num_kv_heads,
                                                     int chunks_per_row, int block_size, long long pool_slots,
                                                     uint32_t *err) {
    pdl_launch_dependents();
    pdl_wait();
    const long long per_token = static_cast<long long>(num_kv_heads) * chunks_per_row;
    const long long total = num_tokens * per_token;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long i = idx / per_token;
        const long long rem = idx - i * per_token;
        const int h = static_cast<int>(rem / chunks_per_row);
        const int c = static_cast<int>(rem - static_cast<long long>(h) * chunks_per_row);
        const long long slot = slots[i];
        if (slot < 0)
            continue;  // padding
        if (slot >= pool_slots) {
            if (err && rem == 0)
                atomicOr(err, PA_DEVERR_BAD_SLOT);
            continue;
        }
        const long long phys = slot / block_size;
        const long long off = slot - phys * block_size;
        const long long dst = ((phys * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
        const uint4 kr = ld_stream(k + idx);
        const uint4 vr = ld_stream(v + idx);
        k_cache[dst] = kr;
        v_cache[dst] = vr;
    }
}

// Quantise-on-append: one warp per (token, kv head) row of K and of V.  Each
// lane holds D / 32 consecutive elements; the row's absolute maximum is a warp
// max, the scale amax / Q is one IEEE fp32 division, and every code is decided
// from the IEEE fp32 quotient x / scale (pa_quant.cuh).  Codes go to the row's
// line of the slot's page as one (D / 32)-byte word per lane (a coalesced
// row), the scale to the page's scale rows (lane 0).
template <int Fmt, int D>
__global__ void __launch_bounds__(256) append_quant_kernel(const char *__restrict__ k, const char *__restrict__ v,
                                                           const int64_t *__restrict__ slots, uint8_t *k_pages,
                                                           uint8_t *v_pages, long long num_tokens, int num_kv_heads,
                                                           int in_dtype, int block_size, long long pool_slots,
                                                           uint32_t *err) {
    constexpr int E = D / 32;
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long rows = num_tokens * num_kv_heads;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const int elt = in_dtype == PA_F32 ? 4 : 2;
    const long long page_bytes = q8_page_bytes(block_size, D);
    for (long long w = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5); w < 2 * rows;
         w += warps) {
        const bool is_v = w >= rows;
        const long long r = is_v ? w - rows : w;  // (token, head) row
        const long long i = r / num_kv_heads;
        const int h = static_cast<int>(r - i * num_kv_heads);
        const long long slot = slots[i];
        if (slot < 0)
            continue;
        if (slot >= pool_slots) {
            if (err && lane == 0 && h == 0 && !is_v)
                atomicOr(err, PA_DEVERR_BAD_SLOT);
            continue;
        }
        const char *src = (is_v ? v : k) + r * D * elt;
        float x[E];
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            x[e] = load_elt(src, in_dtype, lane * E + e);
            amax = fmaxf(amax, fabsf(x[e]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = __fdiv_rn(amax, Q8<Fmt>::kQmax);
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const uint32_t c = s == 0.f ? 0u : Q8<Fmt>::encode(__fdiv_rn(x[e], s));
            word |= c << (8 * e);
        }
        const long long phys = slot / block_size;
        const long long off = slot - phys * block_size;
        uint8_t *page = (is_v ? v_pages : k_pages) + (phys * num_kv_heads + h) * page_bytes;
        uint8_t *codes = page + off * D + lane * E;
        if (E == 4)
            *reinterpret_cast<uint32_t *>(codes) = word;
        else
            *reinterpret_cast<uint16_t *>(codes) = static_cast<uint16_t>(word);
        if (lane == 0)
            reinterpret_cast<float *>(page + static_cast<long long>(block_size) * D)[off] = s;
    }
}

constexpr int kCopyUnroll = 4;

// grid.x: chunks of the block, grid.y: pairs (strided), grid.z: 0 = K, 1 = V.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const int64_t *__restrict__ pairs, int num_pairs,
                                                          uint4 *k_cache, uint4 *v_cache,
                                                          long long chunks_per_block, long long num_blocks,
                                                          uint32_t *err) {
    pdl_launch_dependents();
    pdl_wait();
    uint4 *cache = blockIdx.z == 0 ? k_cache : v_cache;
    for (int pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
        const long long src = pairs[2 * pi], dst = pairs[2 * pi + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (err && blockIdx.x == 0 && threadIdx.x == 0)
                atomicOr(err, PA_DEVERR_BAD_PAIR);
            continue;
        }
        const uint4 *s = cache + src * chunks_per_block;
        uint4 *d = cache + dst * chunks_per_block;
        const long long step = static_cast<long long>(gridDim.x) * blockDim.x * kCopyUnroll;
        for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x * kCopyUnroll + threadIdx.x;
             base < chunks_per_block; base += step) {
            uint4 r[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const long long c = base + static_cast<long long>(u) * blockDim.x;
                if (c < chunks_per_block)
                    r[u] = ld_stream(s + c);
            }
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const long long c = base + static_cast<long long>(u) * blockDim.x;
                if (c < chunks_per_block)
                    d[c] = r[u];
            }
        }
    }
}

// Swap: the same block copy between two pools (device memory, or host memory
// the GPU can address).  grid.x: chunks, grid.y: pairs (strided), grid.z: K / V.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const int64_t *__restrict__ pairs, int num_pairs,
                                                          const uint4 *src_k, const uint4 *src_v, uint4 *dst_k,
                                                          uint4 *dst_v, long long chunks_per_block,
                                                          long long src_blocks, long long dst_blocks, uint32_t *err) {
    pdl_launch_dependents();
    pdl_wait();
    const uint4 *src_pool = blockIdx.z == 0 ? src_k : src_v;
    uint4 *dst_pool = blockIdx.z == 0 ? dst_k : dst_v;
    for (int pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
        const long long src = pairs[2 * pi], dst = pairs[2 * pi + 1];
        if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
            if (err && blockIdx.x == 0 && threadIdx.x == 0)
                atomicOr(err, PA_DEVERR_BAD_PAIR);
            continue;
        }
        const uint4 *s = src_pool + src * chunks_per_block;
        uint4 *d = dst_pool + dst * chunks_per_block;
        const long long step = static_cast<long long>(gridDim.x) * blockDim.x * kCopyUnroll;
        for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x * kCopyUnroll + threadIdx.x;
             base < chunks_per_block; base += step) {
            uint4 r[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const long long c = base + static_cast<long long>(u) * blockDim.x;
                if (c < chunks_per_block)
                    r[u] = ld_stream(s + c);
            }
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const long long c = base + static_cast<long long>(u) * blockDim.x;
                if (c < chunks_per_block)
                    d[c] = r[u];
            }
        }
    }
}

}  // namespace

cudaError_t launch_swap_blocks(const int64_t *pairs, int num_pairs, const void *src_k, const void *src_v,
                               void *dst_k, void *dst_v, long long block_bytes, int src_blocks, int dst_blocks,
                               uint32_t *err, int num_sms, cudaStream_t stream) {
    const long long chunks = block_bytes / 16;
    const long long per_cta = 256LL * kCopyUnroll;
    const long long gx = (chunks + per_cta - 1) / per_cta;
    long long gy = num_pairs;
    const long long cap = static_cast<long long>(num_sms) * 8;  // CTAs in flight for either link's latency
    if (gx * gy * 2 > cap) {
        gy = cap / (2 * gx);
        if (gy < 1)
            gy = 1;
    }
    if (gy > 65535)
        gy = 65535;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 2);
    const uint4 *sk = static_cast<const uint4 *>(src_k), *sv = static_cast<const uint4 *>(src_v);
    uint4 *dk = static_cast<uint4 *>(dst_k), *dv = static_cast<uint4 *>(dst_v);
    long long ck = chunks, sb = src_blocks, db = dst_blocks;
    int np = num_pairs;
    void *args[] = {&pairs, &np, &sk, &sv, &dk, &dv, &ck, &sb, &db, &err};
    return launch_dependent(reinterpret_cast<const void *>(&swap_blocks_kernel), grid, dim3(256), args, 0, stream);
}

cudaError_t launch_append(const void *k, const void *v, const int64_t *slots, void *k_cache, void *v_cache,
                          int num_tokens, int num_kv_heads, int row_bytes, int block_size, int num_blocks,
                          uint32_t *err, int num_sms, cudaStream_t stream) {
    const int cpr = row_bytes / 16;
    const long long total = static_cast<long long>(num_tokens) * num_kv_heads * cpr;
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    const uint4 *ka = static_cast<const uint4 *>(k), *va = static_cast<const uint4 *>(v);
    uint4 *kc = static_cast<uint4 *>(k_cache), *vc = static_cast<uint4 *>(v_cache);
    long long nt = num_tokens, pool_slots = static_cast<long long>(num_blocks) * block_size;
    int hkv = num_kv_heads, c = cpr, bs = block_size;
    void *args[] = {&ka, &va, &slots, &kc, &vc, &nt, &hkv, &c, &bs, &pool_slots, &err};
    return launch_dependent(reinterpret_cast<const void *>(&append_kernel), dim3(static_cast<unsigned>(blocks)),
                            dim3(256), args, 0, stream);
}

cudaError_t launch_append_quant(const void *k, const void *v, const int64_t *slots, void *k_pages, void *v_pages,
                                int num_tokens, int num_kv_heads, int head_dim, int in_dtype, int cache_dtype,
                                int block_size, int num_blocks, uint32_t *err, int num_sms, cudaStream_t stream) {
    const long long warps = 2LL * num_tokens * num_kv_heads;
    long long blocks = (warps + 7) / 8;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    long long pool_slots = static_cast<long long>(num_blocks) * block_size, nt = num_tokens;
    const char *ka = static_cast<const char *>(k), *va = static_cast<const char *>(v);
    uint8_t *kp = static_cast<uint8_t *>(k_pages), *vp = static_cast<uint8_t *>(v_pages);
    int hkv = num_kv_heads, dt = in_dtype, bs = block_size;
    void *args[] = {&ka, &va, &slots, &kp, &vp, &nt, &hkv, &dt, &bs, &pool_slots, &err};
    const void *fn = cache_dtype == PA_I8
                         ? (head_dim == 128 ? reinterpret_cast<const void *>(&append_quant_kernel<kFmtI8, 128>)
                                            : reinterpret_cast<const void *>(&append_quant_kernel<kFmtI8, 64>))
                         : (head_dim == 128 ? reinterpret_cast<const void *>(&append_quant_kernel<kFmtE4M3, 128>)
                                            : reinterpret_cast<const void *>(&append_quant_kernel<kFmtE4M3, 64>));
    return launch_dependent(fn, dim3(static_cast<unsigned>(blocks)), dim3(256), args, 0, stream);
}

cudaError_t launch_copy_blocks(const int64_t *pairs, int num_pairs, void *k_cache, void *v_cache,
                               long long block_bytes, int num_blocks, uint32_t *err, int num_sms,
                               cudaStream_t stream) {
    const long long chunks = block_bytes / 16;
    const long long per_cta = 256LL * kCopyUnroll;
    long long gx = (chunks + per_cta - 1) / per_cta;
    // enough CTAs in flight to cover HBM latency, without exceeding ~8 per SM
    long long gy = num_pairs;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (gx * gy * 2 > cap) {
        gy = cap / (2 * gx);
        if (gy < 1)
            gy = 1;
    }
    if (gy > 65535)
        gy = 65535;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), 2);
    uint4 *kc = static_cast<uint4 *>(k_cache), *vc = static_cast<uint4 *>(v_cache);
    long long ck = chunks, nb = num_blocks;
    int np = num_pairs;
    void *args[] = {&pairs, &np, &kc, &vc, &ck, &nb, &err};
    return launch_dependent(reinterpret_cast<const void *>(&copy_blocks_kernel), grid, dim3(256), args, 0, stream);
}

}  // namespace pa
