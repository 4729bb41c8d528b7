// Paged decode attention for one query head per kv head (MHA): persistent,
// warp-specialised kernel fed by TMA tensor copies.
//
// Computes the same thing as the general decode kernel (pa_decode.cuh):
// softmax(scale * q K^T) V over each sequence's attended tokens, K/V rows
// found through the block table ("PagedAttention — 把 KV cache 当虚拟内存页来管理",
// 案例 2), split into context partitions merged by the log-sum-exp reduce.
//
// What differs is the data path, shaped for HBM bandwidth on sm_103a:
//  - K and V tiles of one (block, kv head) arrive by one 4-D TMA tensor copy
//    each (cp.async.bulk.tensor) in 128-byte-swizzled shared-memory layout: a tile
//    row of d * elt bytes is split into 128-byte boxes whose 16-byte chunks
//    are XOR-permuted by row, so both access patterns below are free of bank
//    conflicts.
//  - Items (sequence, kv head, partition) flow through a small ring filled by
//    the producer warp (item_full / item_empty mbarriers); each item's query
//    row rides on the item_full barrier.  The pipeline stages (one cache
//    block each) form one sub-ring per consumer warp, and block j of every
//    item goes to warp j % 4: a warp waits only for its own blocks, and which
//    warp sums which blocks does not depend on the items a CTA ran before,
//    so the result is the same bits on every run.
//  - QK: lanes are (part, token) pairs — 16 tokens per round (8 at block size
//    8), each token's row split over 32 / 16 (or 32 / 8) lanes — and every
//    lane accumulates its share of the dot product with mixed-precision FMA
//    (fp16/bf16 operands, fp32 accumulate; products are exact), then one or
//    two shuffles finish each score.
//  - Softmax: per round one max over the round's tokens, a rescale of the
//    running state only when the max grows, p = 2^(s - m).
//  - PV: each lane owns head_dim / 32 output dimensions and accumulates
//    p_t * v_t[dims] in fp32, p_t broadcast by a shuffle.
// Every wait is bounded (PA_DEVERR_TIMEOUT); bad table entries are never
// dereferenced (PA_DEVERR_BAD_BLOCK).
#pragma once

#include <cuda.h>  // CUtensorMap (type only)

#include "pa_decode.cuh"

namespace pa {

constexpr int kMhaWarps = 4;
constexpr int kMhaNearBlocks = 8;  // blocks of an item still to issue when the next item is claimed
constexpr int kMhaThreads = (kMhaWarps + 1) * 32;
constexpr int kItemSlots = 4;

struct MhaItem {
    int s, kvh, part, nparts;
    int nb;        // blocks of the item (0: empty sequence)
    int tok_lo;    // attended tokens of the item: [tok_lo, tok_hi)
    int tok_hi;
    int blk_lo;    // first logical block
    int t_first;   // pipeline stage of the first block
    int end;       // 1: no more items
    int pad[2];
};

template <typename T, int D, int BS> struct MhaCfg {
    static constexpr int kElt = sizeof(T);
    static constexpr int kRow = D * kElt;              // bytes per token row
    static constexpr int kBoxes = kRow / 128;          // 128-byte swizzle boxes per row
    static constexpr int kTile = BS * kRow;
    static constexpr int kTpr = BS < 16 ? BS : 16;     // tokens per QK round
    static constexpr int kRounds = BS / kTpr;
    static constexpr int kLpt = 32 / kTpr;             // lanes per token in QK
    static constexpr int kChunks = kRow / 16;          // 16-byte chunks per row
    static constexpr int kCpl = kChunks / kLpt;        // QK chunks per lane
    static constexpr int kDpl = D / 32;                // PV dimensions per lane
    static constexpr int kPvBytes = kDpl * kElt;       // PV bytes per lane per token
    static_assert(kBoxes >= 1 && kRow % 128 == 0, "rows must be whole 128-byte boxes");
    static_assert(kCpl >= 1 && kChunks % kLpt == 0, "row chunks must split evenly over a token's lanes");
    static_assert(kPvBytes == 4 || kPvBytes == 8 || kPvBytes == 16, "PV load width");
};

struct MhaLayout {
    uint32_t full, empty, ifull, iempty, mfull, mempty, valid, items, table, qbuf, mscr, mml, stages, total;
};

__host__ __device__ inline MhaLayout mha_smem_layout(int S, int tile_bytes, int row_bytes, int D) {
    MhaLayout L;
    uint32_t off = 0;
    L.full = off;
    off += 8 * S;
    L.empty = off;
    off += 8 * S;
    L.ifull = off;
    off += 8 * kItemSlots;
    L.iempty = off;
    off += 8 * kItemSlots;
    L.mfull = off;
    off += 16;
    L.mempty = off;
    off += 16;
    L.valid = off;
    off += 4 * S;
    L.items = align_up(off, 16);
    off = L.items + sizeof(MhaItem) * kItemSlots;
    L.table = off;
    off += 4 * kMaxBpp;
    L.qbuf = align_up(off, 128);
    off = L.qbuf + kItemSlots * row_bytes;
    L.mscr = align_up(off, 16);
    off = L.mscr + 2 * kMhaWarps * D * 4;
    L.mml = off;
    off += 2 * kMhaWarps * 2 * 4;
    L.stages = align_up(off, 1024);  // 128-byte swizzle repeats every 1024 bytes
    off = L.stages + S * 2 * tile_bytes;
    L.total = off + 1024;  // slack to align the dynamic shared memory base
    return L;
}

// ---------------------------------------------------------------------------
// PTX helpers specific to this kernel

// One whole (block, head) tile through the 4-D view
// [tile][128-byte segment][row][segment elements]: kBoxes boxes of block_size
// rows x 128 bytes, back to back.
__device__ inline void tma_load_4d(void *dst, const CUtensorMap *map, int z, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(0), "r"(z), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ inline void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ inline float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// acc += sum of the elementwise products of two 16-byte chunks (fp32 accumulate).
template <typename T> struct ChunkDot;
template <> struct ChunkDot<__half> {
    __device__ static inline void run(const uint4 &q, const uint4 &k, float &a0, float &a1) {
        asm("{\n\t.reg .b16 x0, x1, y0, y1;\n\t"
            "mov.b32 {x0, x1}, %2;\n\tmov.b32 {y0, y1}, %6;\n\t"
            "fma.rn.f32.f16 %0, x0, y0, %0;\n\tfma.rn.f32.f16 %1, x1, y1, %1;\n\t"
            "mov.b32 {x0, x1}, %3;\n\tmov.b32 {y0, y1}, %7;\n\t"
            "fma.rn.f32.f16 %0, x0, y0, %0;\n\tfma.rn.f32.f16 %1, x1, y1, %1;\n\t"
            "mov.b32 {x0, x1}, %4;\n\tmov.b32 {y0, y1}, %8;\n\t"
            "fma.rn.f32.f16 %0, x0, y0, %0;\n\tfma.rn.f32.f16 %1, x1, y1, %1;\n\t"
            "mov.b32 {x0, x1}, %5;\n\tmov.b32 {y0, y1}, %9;\n\t"
            "fma.rn.f32.f16 %0, x0, y0, %0;\n\tfma.rn.f32.f16 %1, x1, y1, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w), "r"(k.x), "r"(k.y), "r"(k.z), "r"(k.w));
    }
};
template <> struct ChunkDot<__nv_bfloat16> {
    __device__ static inline void run(const uint4 &q, const uint4 &k, float &a0, float &a1) {
        asm("{\n\t.reg .b16 x0, x1, y0, y1;\n\t"
            "mov.b32 {x0, x1}, %2;\n\tmov.b32 {y0, y1}, %6;\n\t"
            "fma.rn.f32.bf16 %0, x0, y0, %0;\n\tfma.rn.f32.bf16 %1, x1, y1, %1;\n\t"
            "mov.b32 {x0, x1}, %3;\n\tmov.b32 {y0, y1}, %7;\n\t"
            "fma.rn.f32.bf16 %0, x0, y0, %0;\n\tfma.rn.f32.bf16 %1, x1, y1, %1;\n\t"
            "mov.b32 {x0, x1}, %4;\n\tmov.b32 {y0, y1}, %8;\n\t"
            "fma.rn.f32.bf16 %0, x0, y0, %0;\n\tfma.rn.f32.bf16 %1, x1, y1, %1;\n\t"
            "mov.b32 {x0, x1}, %5;\n\tmov.b32 {y0, y1}, %9;\n\t"
            "fma.rn.f32.bf16 %0, x0, y0, %0;\n\tfma.rn.f32.bf16 %1, x1, y1, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w), "r"(k.x), "r"(k.y), "r"(k.z), "r"(k.w));
    }
};
template <> struct ChunkDot<float> {
    __device__ static inline void run(const uint4 &q, const uint4 &k, float &a0, float &a1) {
        a0 = fmaf(__uint_as_float(q.x), __uint_as_float(k.x), a0);
        a1 = fmaf(__uint_as_float(q.y), __uint_as_float(k.y), a1);
        a0 = fmaf(__uint_as_float(q.z), __uint_as_float(k.z), a0);
        a1 = fmaf(__uint_as_float(q.w), __uint_as_float(k.w), a1);
    }
};

// Load the PV slice (kPvBytes) of one V row and widen it to fp32.
template <typename T, int N> struct PvLoad;
template <> struct PvLoad<__half, 4> {  // d 128
    __device__ static inline void run(const char *p, float *v) {
        const uint2 r = ld_shared_v2(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
        v[0] = a.x, v[1] = a.y, v[2] = b.x, v[3] = b.y;
    }
};
template <> struct PvLoad<__half, 2> {  // d 64
    __device__ static inline void run(const char *p, float *v) {
        const uint32_t r = ld_shared_u32(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r));
        v[0] = a.x, v[1] = a.y;
    }
};
template <> struct PvLoad<__nv_bfloat16, 4> {
    __device__ static inline void run(const char *p, float *v) {
        const uint2 r = ld_shared_v2(p);
        v[0] = __uint_as_float(r.x << 16), v[1] = __uint_as_float(r.x & 0xffff0000u);
        v[2] = __uint_as_float(r.y << 16), v[3] = __uint_as_float(r.y & 0xffff0000u);
    }
};
template <> struct PvLoad<__nv_bfloat16, 2> {
    __device__ static inline void run(const char *p, float *v) {
        const uint32_t r = ld_shared_u32(p);
        v[0] = __uint_as_float(r << 16), v[1] = __uint_as_float(r & 0xffff0000u);
    }
};
template <> struct PvLoad<float, 4> {
    __device__ static inline void run(const char *p, float *v) {
        const uint4 r = ld_shared_v4(p);
        v[0] = __uint_as_float(r.x), v[1] = __uint_as_float(r.y), v[2] = __uint_as_float(r.z),
        v[3] = __uint_as_float(r.w);
    }
};
template <> struct PvLoad<float, 2> {
    __device__ static inline void run(const char *p, float *v) {
        const uint2 r = ld_shared_v2(p);
        v[0] = __uint_as_float(r.x), v[1] = __uint_as_float(r.y);
    }
};

// Byte offset of (row r, 16-byte chunk c of the whole row) inside a swizzled tile.
template <int BS>
__device__ inline uint32_t swz(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * (BS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------------------

template <typename T, int D, int BS>
__device__ inline void mha_producer(const DecodeParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                    char *smem, const MhaLayout &L) {
    using C = MhaCfg<T, D, BS>;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    int *valid = reinterpret_cast<int *>(smem + L.valid);
    MhaItem *items = reinterpret_cast<MhaItem *>(smem + L.items);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + L.table);
    char *qbuf = smem + L.qbuf;
    char *stage_buf = smem + L.stages;
    const char *qg = static_cast<const char *>(p.q);
    const uint64_t policy = policy_evict_first();
    if (lane == 0) {
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
    }

    ItemScan scan;
    // blocks issued into each consumer warp's sub-ring of S / 4 stages
    uint32_t cw[kMhaWarps] = {0, 0, 0, 0};
    const int S4 = S / kMhaWarps;
    int k = 0;  // items issued
    bool ok = true;
    const long long hkv = p.num_kv_heads;

    ItemClaim claim;
    // the next item is claimed when the current one has kMhaNearBlocks blocks
    // left to issue, so the launch's last items go to the CTAs that run out first
    claim.start();
    for (;; claim.next(p)) {
        const long long w = claim.w;
        const long long f = w / hkv;
        const int kvh = static_cast<int>(w % hkv);
        int part = 0, len = 0, start = 0;
        const int s = scan.find(p, BS, f, part, len, start);

        const int slot = k % kItemSlots;
        if (!mbar_wait_bounded(&iempty[slot], ((k / kItemSlots) & 1) ^ 1)) {
            ok = false;
            break;
        }
        if (s < 0) {  // no more items: publish the end marker
            if (lane == 0) {
                items[slot].end = 1;
                mbar_arrive(&ifull[slot]);
            }
            __syncwarp();
            break;
        }
        const SeqSpan sp = seq_span(len, p.max_len, p.window, BS, p.bpp, start);
        const int blk_lo = sp.b0 + part * p.bpp;
        const int nb = max(0, min(p.bpp, sp.nblk - part * p.bpp));
        if (lane == 0) {
            MhaItem it;
            it.s = s;
            it.kvh = kvh;
            it.part = part;
            it.nparts = sp.nparts;
            it.nb = nb;
            it.tok_lo = max(sp.start, blk_lo * BS);
            it.tok_hi = min(sp.end, (blk_lo + nb) * BS);
            it.blk_lo = blk_lo;
            it.t_first = 0;  // (stages follow from the block index: sub-ring j % 4)
            it.end = 0;
            items[slot] = it;
            if (nb > 0) {
                mbar_arrive_expect_tx(&ifull[slot], C::kRow);
                bulk_g2s(qbuf + slot * C::kRow, qg + (static_cast<long long>(s) * p.num_heads + kvh) * C::kRow,
                         C::kRow, &ifull[slot]);
            } else {
                mbar_arrive(&ifull[slot]);
            }
        }
        // block-table slice of the item -> shared memory, entries range-checked
        const int32_t *row = p.block_tables + static_cast<long long>(s) * p.max_blocks_per_seq + blk_lo;
        for (int j = lane; j < nb; j += 32) {
            int pb = p.contiguous ? blk_lo + j : ld_nc_i32(row + j);
            if (pb < 0 || pb >= p.num_blocks) {
                pb = -1;
                if (p.err)
                    atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
            }
            tbl[j] = pb;
        }
        __syncwarp();
        for (int j0 = 0; j0 < nb && ok; j0 += kMhaWarps) {
#pragma unroll
            for (int w = 0; w < kMhaWarps; ++w) {
            const int j = j0 + w;
            if (j >= nb)
                break;
            if (j == max(0, nb - kMhaNearBlocks))
                claim.claim_next(p);
            const uint32_t c = cw[w]++;
            const int stage = w * S4 + static_cast<int>(c % S4);
            if (!mbar_wait_bounded(&empty[stage], ((c / S4) & 1u) ^ 1u)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const int pb = tbl[j];
                valid[stage] = pb >= 0;
                if (pb >= 0) {
                    mbar_arrive_expect_tx(&full[stage], 2 * C::kTile);
                    char *dk = stage_buf + static_cast<size_t>(stage) * 2 * C::kTile;
                    char *dv = dk + C::kTile;
                    const int z = kv_tile(p, s, kvh, pb);
                    tma_load_4d(dk, tmk, z, &full[stage], policy);
                    tma_load_4d(dv, tmv, z, &full[stage], policy);
                } else {
                    mbar_arrive(&full[stage]);
                }
            }
            __syncwarp();
            }
        }
        if (!ok)
            break;
        ++k;
    }
    if (!ok && lane == 0) {
        // a wait gave up: flag it, then wait (bounded) for our copies in flight
        if (p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
#pragma unroll
        for (int w = 0; w < kMhaWarps; ++w) {
            const uint32_t first = cw[w] > static_cast<uint32_t>(S4) ? cw[w] - S4 : 0;
            for (uint32_t u = first; u < cw[w]; ++u)
                (void)mbar_wait_bounded(&full[w * S4 + static_cast<int>(u % S4)], (u / S4) & 1u);
        }
    }
    claim.finish(p);
    __syncwarp();
}

template <typename T, int D, int BS>
__device__ inline void mha_consumer(const DecodeParams &p, char *smem, const MhaLayout &L) {
    using C = MhaCfg<T, D, BS>;
    constexpr int kDpl = C::kDpl;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tok = lane % C::kTpr;    // QK: token of the round
    const int part = lane / C::kTpr;   // QK: share of the row
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint64_t *mfull = reinterpret_cast<uint64_t *>(smem + L.mfull);
    uint64_t *mempty = reinterpret_cast<uint64_t *>(smem + L.mempty);
    const int *valid = reinterpret_cast<const int *>(smem + L.valid);
    const MhaItem *items = reinterpret_cast<const MhaItem *>(smem + L.items);
    const char *qbuf = smem + L.qbuf;
    float *mscr = reinterpret_cast<float *>(smem + L.mscr);  // [2][warps][D]
    float *mml = reinterpret_cast<float *>(smem + L.mml);    // [2][warps][2]
    const char *stage_buf = smem + L.stages;

    // PV: byte offset of this lane's slice inside a row (box, chunk, sub-chunk)
    const int pv_off = lane * C::kPvBytes;
    const int pv_chunk = pv_off >> 4;
    const int pv_sub = pv_off & 15;

    uint4 q[C::kCpl];
    bool ok = true;
    const int S4 = S / kMhaWarps;
    uint32_t c = 0;  // blocks this warp took from its sub-ring
    for (int k = 0;; ++k) {
        const int slot = k % kItemSlots;
        if (!mbar_wait_bounded(&ifull[slot], (k / kItemSlots) & 1)) {
            ok = false;
            break;
        }
        const MhaItem it = items[slot];
        if (it.end)
            break;
        if (it.nb > 0) {
#pragma unroll
            for (int i = 0; i < C::kCpl; ++i)
                q[i] = ld_shared_v4(qbuf + slot * C::kRow + (part * C::kCpl + i) * 16);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&iempty[slot]);

        float m = -INFINITY, l = 0.f;
        float acc[kDpl];
#pragma unroll
        for (int i = 0; i < kDpl; ++i)
            acc[i] = 0.f;

        for (int j = warp; j < it.nb; j += kMhaWarps, ++c) {
            const int stage = warp * S4 + static_cast<int>(c % S4);
            if (!mbar_wait_bounded(&full[stage], (c / S4) & 1u)) {
                ok = false;
                break;
            }
            if (valid[stage]) {
                const char *kt = stage_buf + static_cast<size_t>(stage) * 2 * C::kTile;
                const char *vt = kt + C::kTile;
                const int blk = it.blk_lo + j;
                const int lo = max(it.tok_lo - blk * BS, 0);
                const int hi = min(it.tok_hi - blk * BS, BS);
#pragma unroll
                for (int rd = 0; rd < C::kRounds; ++rd) {
                    const int r0 = rd * C::kTpr;
                    if (r0 >= hi || r0 + C::kTpr <= lo)
                        continue;
                    // scores of this round's tokens
                    const int r = r0 + tok;
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int i = 0; i < C::kCpl; ++i)
                        ChunkDot<T>::run(q[i], ld_shared_v4(kt + swz<BS>(r, part * C::kCpl + i)), a0, a1);
                    float sc = a0 + a1;
#pragma unroll
                    for (int o = C::kTpr; o < 32; o <<= 1)
                        sc += __shfl_xor_sync(0xffffffffu, sc, o);
                    sc = (r >= lo && r < hi) ? sc * p.scale_log2 : -INFINITY;
                    float mr = sc;
#pragma unroll
                    for (int o = 1; o < C::kTpr; o <<= 1)
                        mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
                    if (mr > m) {  // the running max grows: rescale the state
                        const float alpha = fast_exp2(m - mr);
                        l *= alpha;
#pragma unroll
                        for (int i = 0; i < kDpl; ++i)
                            acc[i] *= alpha;
                        m = mr;
                    }
                    const float pw = fast_exp2(sc - m);
                    if (part == 0)
                        l += pw;
                    // P V over the round's attended tokens
                    const int t_lo = max(lo - r0, 0), t_hi = min(hi - r0, C::kTpr);
#pragma unroll
                    for (int u = 0; u < C::kTpr; ++u) {
                        const float pu = __shfl_sync(0xffffffffu, pw, u);
                        if (u >= t_lo && u < t_hi) {
                            float v[kDpl];
                            PvLoad<T, kDpl>::run(vt + swz<BS>(r0 + u, pv_chunk) + pv_sub, v);
#pragma unroll
                            for (int i = 0; i < kDpl; ++i)
                                acc[i] = fmaf(pu, v[i], acc[i]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
        }
        if (!ok)
            break;

        // merge the 4 warps' states of this item (double-buffered by item parity)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            l += __shfl_xor_sync(0xffffffffu, l, o);
        const int b = k & 1;
        const uint32_t use = static_cast<uint32_t>(k >> 1) & 1u;
        if (!mbar_wait_bounded(&mempty[b], use ^ 1u)) {
            ok = false;
            break;
        }
#pragma unroll
        for (int i = 0; i < kDpl; ++i)
            mscr[(b * kMhaWarps + warp) * D + lane * kDpl + i] = acc[i];
        if (lane == 0) {
            mml[(b * kMhaWarps + warp) * 2] = m;
            mml[(b * kMhaWarps + warp) * 2 + 1] = l;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&mfull[b]);
        if (!mbar_wait_bounded(&mfull[b], use)) {
            ok = false;
            break;
        }
        float M = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < kMhaWarps; ++w2)
            M = fmaxf(M, mml[(b * kMhaWarps + w2) * 2]);
        float scl[kMhaWarps];
        float den = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kMhaWarps; ++w2) {
            const float mw = mml[(b * kMhaWarps + w2) * 2];
            scl[w2] = (M == -INFINITY) ? 0.f : fast_exp2(mw - M);
            den = fmaf(mml[(b * kMhaWarps + w2) * 2 + 1], scl[w2], den);
        }
        const long long rowi = static_cast<long long>(it.s) * p.num_heads + it.kvh;
        for (int dd = warp * 32 + lane; dd < D; dd += kMhaWarps * 32) {
            float num = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kMhaWarps; ++w2)
                num = fmaf(mscr[(b * kMhaWarps + w2) * D + dd], scl[w2], num);
            if (it.nparts == 1 && !p.force_partial) {
                store_out(p.out, p.out_dtype, rowi * D + dd, den > 0.f ? num / den : 0.f);
            } else {
                const long long pr = rowi * p.max_parts + it.part;
                p.part_acc[pr * D + dd] = num;
                if (dd == 0) {
                    p.part_ml[pr * 2] = M;
                    p.part_ml[pr * 2 + 1] = den;
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&mempty[b]);
    }
    if (!ok && lane == 0 && p.err)
        atomicOr(p.err, PA_DEVERR_TIMEOUT);
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kMhaThreads) pa_decode_mha_kernel(const DecodeParams p,
                                                                   const __grid_constant__ CUtensorMap tmk,
                                                                   const __grid_constant__ CUtensorMap tmv) {
    // the next kernel on the stream may be launched now (it waits for this
    // grid); this one waits for the kernel before it
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using C = MhaCfg<T, D, BS>;
    const MhaLayout L = mha_smem_layout(p.stages, C::kTile, C::kRow, D);
    // The stages are one sub-ring of S / 4 per consumer warp: S must be a
    // multiple of 4.  The host never launches another count; refuse it here too.
    if (p.stages < kMhaWarps || p.stages % kMhaWarps != 0) {
        if (threadIdx.x == 0 && p.err)
            atomicOr(p.err, PA_DEVERR_BAD_LAUNCH);
        return;
    }
    if (threadIdx.x == 0) {
        uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
        uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
        uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(&ifull[i], 1);
            mbar_init(&iempty[i], kMhaWarps);
        }
        uint64_t *mfull = reinterpret_cast<uint64_t *>(smem + L.mfull);
        uint64_t *mempty = reinterpret_cast<uint64_t *>(smem + L.mempty);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&mfull[i], kMhaWarps);
            mbar_init(&mempty[i], kMhaWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if ((threadIdx.x >> 5) == kMhaWarps)
        mha_producer<T, D, BS>(p, &tmk, &tmv, smem, L);
    else
        mha_consumer<T, D, BS>(p, smem, L);
    __syncthreads();
    release_claims(p);
}

}  // namespace pa
