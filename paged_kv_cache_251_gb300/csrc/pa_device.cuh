// Device-side helpers shared by the kernels of libpa: PTX wrappers for
// mbarriers and bulk (TMA) copies, bounded waits, element conversion and the
// context-partition arithmetic that the decode and reduce kernels must agree on.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------------------
// Element types

template <typename T> struct Elt;
template <> struct Elt<float> {
    static constexpr int kCode = PA_F32;
    __device__ static inline void unpack(const uint4 &r, float *f) {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z);
        f[3] = __uint_as_float(r.w);
    }
};
template <> struct Elt<__half> {
    static constexpr int kCode = PA_F16;
    __device__ static inline void unpack(const uint4 &r, float *f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 p = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
};
template <> struct Elt<__nv_bfloat16> {
    static constexpr int kCode = PA_BF16;
    __device__ static inline void unpack(const uint4 &r, float *f) {
        // bf16 is the top half of an fp32: widening is a shift / mask.
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

__device__ inline void store_out(void *out, int dtype, int64_t idx, float v) {
    if (dtype == PA_F32)
        static_cast<float *>(out)[idx] = v;
    else if (dtype == PA_F16)
        static_cast<__half *>(out)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------------------
// PTX wrappers

__device__ inline uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch: a decode kernel lets the kernel that merges
// its partials be launched while it runs (launch_dependents, once per CTA at
// its start); that kernel, launched with programmatic stream serialization,
// waits for the whole decode grid and its memory (wait) before it reads
// anything.  Both are no-ops without such a launch.
__device__ inline void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ inline uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ inline void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ inline void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ inline void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ inline bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// A wait that gives up: every wait in these kernels ends, either because the
// phase completed or because about kTimeoutNs passed (the caller then flags
// PA_DEVERR_TIMEOUT and winds down).
constexpr uint64_t kTimeoutNs = 2000000000ull;

__device__ inline bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 15u) == 0 && globaltimer_ns() - t0 > kTimeoutNs)
            return false;
    }
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ inline void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same, with an L2 eviction-priority policy (streamed K/V is read once).
__device__ inline void bulk_g2s_hint(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar,
                                     uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ inline uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ inline uint2 ld_shared_v2(const void *p) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(smem_addr(p)));
    return r;
}

__device__ inline uint32_t ld_shared_u32(const void *p) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(smem_addr(p)));
    return r;
}

__device__ inline uint4 ld_shared_v4(const void *p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_addr(p)));
    return r;
}

__device__ inline int ld_nc_i32(const int32_t *p) {
    int v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// Context partitions.  The attended tokens of sequence s are
// [start, L) with start = max(0, L - window) when window > 0.  Partitions
// are aligned to the block grid: partition p covers logical blocks
// [b0 + p * bpp, b0 + (p + 1) * bpp) with b0 = start / block_size, clipped to
// the attended tokens, so no block is read by two partitions.  A sequence
// with no attended token still has one (empty) partition, which writes zeros.

struct SeqSpan {
    int start;   // first attended token
    int end;     // one past the last attended token (= L)
    int b0;      // first logical block
    int nblk;    // logical blocks touched
    int nparts;  // >= 1
};

// max_len = max_blocks_per_seq * block_size: a longer context would index past
// the table row, so it is clamped (and the caller flags PA_DEVERR_BAD_LEN).
// start_min (0 normally) moves the first attended token further up: the
// shared-prefix decode uses it for the part of a context after the prefix.
__device__ inline SeqSpan seq_span(int L, int max_len, int window, int block_size, int bpp, int start_min = 0) {
    SeqSpan sp;
    if (L < 0)
        L = 0;
    if (L > max_len)
        L = max_len;
    sp.end = L;
    sp.start = (window > 0 && L > window) ? L - window : 0;
    if (start_min > sp.start)
        sp.start = start_min < L ? start_min : L;
    sp.b0 = sp.start / block_size;
    sp.nblk = L > sp.start ? (L - 1) / block_size - sp.b0 + 1 : 0;
    sp.nparts = sp.nblk > 0 ? (sp.nblk + bpp - 1) / bpp : 1;
    return sp;
}

}  // namespace pa
