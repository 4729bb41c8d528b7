// Paged decode attention for grouped-query heads on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// Same result as the other decode kernels: for each sequence and query head,
// softmax(scale * q K^T) V over the attended tokens, K/V rows reached through
// the block table ("PagedAttention — 把 KV cache 当虚拟内存页来管理", 案例 2),
// long contexts split into partitions merged by the log-sum-exp reduce.
//
// With G = num_heads / num_kv_heads query heads sharing one kv head, the two
// products of a 128-token tile are small dense contractions:
//   S  = K  . Q^T   M = 128 tokens,  N = 16 (G heads, rest zero), K = head_dim
//   O^T = V^T . P   M = 128 (head_dim), N = 16 (G heads x {hi, lo}), K = tokens
// Both run as tcgen05.mma kind::f16 (bf16 or fp16 operands, fp32
// accumulate) into tensor memory.  P is split into two 16-bit parts
// (hi = round(p), lo = round(p - hi)) that occupy the N columns the heads
// leave free, so the PV product keeps about 16 mantissa bits of p.
//
// Warp roles (224 threads, one CTA per SM, persistent over items
// (sequence, kv head, partition)):
//   warp 0      K producer: item ring (+ the item's G query rows by TMA),
//               block-table slice into shared memory (range-checked), K of
//               each 128-token tile by 5-D TMA tensor copies (one per block,
//               issued by one lane per block; 128-byte swizzle) into the K
//               half of a ring of stages, and a record per stage of the
//               tile's blocks for the V producer;
//   warp 6      V producer: V of each tile into the V half of its stage, from
//               the record.  The two halves are released separately: K once
//               S of its tile finished (and the softmax warps read the
//               tile's block mask), V once P V finished.  A stage's K half
//               is thus refilled while its V is still in use, which keeps
//               more of the ring in flight: the kernel is bound by the bytes
//               each SM keeps in flight to HBM;
//   warp 1      tensor-memory allocation and the single thread that issues
//               the MMAs and their commits; tile g's S = K . Q^T is issued
//               before tile g-1's P V, so scoring overlaps the P V product;
//   warps 2..5  softmax and epilogue.  Each warp owns one quarter of every
//               tile's tokens (its tensor-memory lane quarter) with its own
//               running max and denominator per head, so no cross-warp step
//               sits on the per-tile path; P V is one accumulator per quarter,
//               and the epilogue (one thread per head_dim row) keeps one running
//               output per quarter, merged once per item.
// Every wait is bounded (PA_DEVERR_TIMEOUT); tensor memory is freed on every
// path; bad table entries are never dereferenced (PA_DEVERR_BAD_BLOCK).
#pragma once

#include <type_traits>

#include "pa_decode_mha.cuh"

namespace pa {

constexpr int kGqaThreads = 7 * 32;
constexpr int kGqaSmWarps = 4;    // softmax / epilogue warps
constexpr int kGqaItemSlots = 4;
constexpr int kGqaNearTiles = 4;  // tiles of an item still to issue when the next item is claimed
constexpr int kTileTokens = 128;  // MMA M
constexpr int kTmemCols = 256;    // S[2] (16 cols) at 0..31, O[2][4 quarters] (16 cols) at 32..159

template <typename T, int BS, int G> struct GqaCfg {
    static constexpr int kD = 128;
    static constexpr int kElt = 2;
    static constexpr int kRow = kD * kElt;               // 256 bytes
    static constexpr int kBpt = kTileTokens / BS;        // blocks per tile
    // K (or V) of one tile: [token / 8][half of head_dim][token % 8][128 B],
    // i.e. 8-row groups of 2 KB, each holding both 64-column halves
    static constexpr int kGroupBytes = 2048;
    static constexpr int kHalfBytes = 1024;
    static constexpr int kTile = kTileTokens / 8 * kGroupBytes;  // 32 KB
    static constexpr int kBlockBytes = BS * kRow;                // one block: all rows, both halves
    static constexpr int kOpBytes = 2 * 16 * 128;        // Q or P operand: 2 boxes x 16 rows x 128 B
    static constexpr uint32_t kFullMask = (1u << kBpt) - 1u;  // every block of a tile
    static_assert(sizeof(T) == 2, "tensor-core path takes 16-bit K/V");
    static_assert(G == 2 || G == 4 || G == 8, "query group");
};

struct GqaLayout {
    uint32_t kfull, vfull, kempty, vempty, zfull, zfree, ifull, iempty, sfull, sfree, pfull, ofull, ofree, xfull, done,
        fin;
    uint32_t meta, zmask, zid, items, tmem, table, xbuf, abuf, qbuf, pbuf, stages, total;
};

// The V producer's record of a stage: the valid-block mask of its tile (or
// this value: no more tiles) and the blocks' tensor-map tile indices.
constexpr uint32_t kGqaEndRecord = 0xFFFFFFFFu;
constexpr int kGqaMaxBpt = 16;  // blocks per 128-token tile at block size 8

__host__ __device__ inline GqaLayout gqa_smem_layout(int S) {
    GqaLayout L;
    uint32_t off = 0;
    L.kfull = off;
    off += 8 * S;
    L.vfull = off;
    off += 8 * S;
    L.kempty = off;
    off += 8 * S;
    L.vempty = off;
    off += 8 * S;
    L.zfull = off;
    off += 8 * S;
    L.zfree = off;
    off += 8 * S;
    L.ifull = off;
    off += 8 * kGqaItemSlots;
    L.iempty = off;
    off += 8 * kGqaItemSlots;
    L.sfull = off;
    off += 16;
    L.sfree = off;
    off += 16;
    L.pfull = off;
    off += 16;
    L.ofull = off;
    off += 16;
    L.ofree = off;
    off += 16;
    L.xfull = off;
    off += 16;
    L.done = off;
    off += 8;
    L.fin = off;
    off += 8;
    L.meta = off;
    off += 4 * S;
    L.zmask = off;
    off += 4 * S;
    L.zid = off;
    off += 4 * S * kGqaMaxBpt;
    L.items = align_up(off, 16);
    off = L.items + sizeof(MhaItem) * kGqaItemSlots;
    L.tmem = off;
    off += 16;
    L.table = off;
    off += 4 * kMaxBpp;
    L.xbuf = off;
    off += 2 * kGqaSmWarps * 16 * 4;
    L.abuf = off;
    off += 4 * kGqaSmWarps * 8 * 4;
    L.qbuf = align_up(off, 1024);
    off = L.qbuf + kGqaItemSlots * 2 * 16 * 128;
    L.pbuf = off;
    off += 2 * 2 * 16 * 128;
    L.stages = align_up(off, 1024);
    off = L.stages + S * 2 * (2 * kTileTokens * 128);
    L.total = off + 1024;
    return L;
}

// ---------------------------------------------------------------------------
// tcgen05 / TMA wrappers

__device__ inline void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ inline void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ inline void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ inline void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ inline void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ inline void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ inline void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ inline void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int N> __device__ inline void tmem_ld(uint32_t taddr, float *v);
template <> __device__ inline void tmem_ld<2>(uint32_t taddr, float *v) {
    uint32_t r0, r1;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(taddr));
    v[0] = __uint_as_float(r0), v[1] = __uint_as_float(r1);
}
template <> __device__ inline void tmem_ld<4>(uint32_t taddr, float *v) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = __uint_as_float(r[i]);
}
template <> __device__ inline void tmem_ld<8>(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = __uint_as_float(r[i]);
}
template <> __device__ inline void tmem_ld<16>(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}
__device__ inline void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// One block of one kv head through the 5-D view [tile][row / 8][half][row % 8][64]
// (box = the whole block), landing as 8-row groups of both halves.
__device__ inline void tma_load_5d(void *dst, const CUtensorMap *map, int z, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(0), "r"(0), "r"(z), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

__device__ inline void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format: start
// address, leading / stride byte offsets in 16-byte units, version 1).
__device__ inline uint64_t sdesc(const void *p, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((smem_addr(p) & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulate, A/B element type
// (0 = fp16, 1 = bf16), A/B major-ness (0 = K-major, 1 = MN-major), N and M.
template <typename T>
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn_major, int b_mn_major) {
    return (1u << 4) | ((std::is_same<T, __half>::value ? 0u : 1u) << 7) |
           ((std::is_same<T, __half>::value ? 0u : 1u) << 10) | (static_cast<uint32_t>(a_mn_major) << 15) |
           (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

template <typename T> __device__ inline uint16_t to_bits16(float x);
template <> __device__ inline uint16_t to_bits16<__nv_bfloat16>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <> __device__ inline uint16_t to_bits16<__half>(float x) { return __half_as_ushort(__float2half_rn(x)); }
template <typename T> __device__ inline float from_bits16(uint16_t b);
template <> __device__ inline float from_bits16<__nv_bfloat16>(uint16_t b) {
    return __bfloat162float(__ushort_as_bfloat16(b));
}
template <> __device__ inline float from_bits16<__half>(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// ---------------------------------------------------------------------------

template <typename T, int BS, int G>
__device__ inline void gqa_producer(const DecodeParams &p, const CUtensorMap *tmk, const CUtensorMap *tmkw,
                                    const CUtensorMap *tmq, char *smem, const GqaLayout &L) {
    using C = GqaCfg<T, BS, G>;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + L.kfull);
    uint64_t *kempty = reinterpret_cast<uint64_t *>(smem + L.kempty);
    uint64_t *zfull = reinterpret_cast<uint64_t *>(smem + L.zfull);
    uint64_t *zfree = reinterpret_cast<uint64_t *>(smem + L.zfree);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint32_t *meta = reinterpret_cast<uint32_t *>(smem + L.meta);
    uint32_t *zmask = reinterpret_cast<uint32_t *>(smem + L.zmask);
    int32_t *zid = reinterpret_cast<int32_t *>(smem + L.zid);
    MhaItem *items = reinterpret_cast<MhaItem *>(smem + L.items);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + L.table);
    char *qbuf = smem + L.qbuf;
    char *stage_buf = smem + L.stages;
    const uint64_t policy = policy_evict_first();
    if (lane == 0) {
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmq);
    }
    ItemScan scan;
    uint32_t t = 0;
    bool ok = true;
    const long long hkv = p.num_kv_heads;

    // the next item is claimed (and its table slice loaded) when the current
    // one has kGqaNearTiles tiles left to issue, so the launch's last items go
    // to the CTAs that run out of work first
    ItemClaim claim;
    claim.start();
    NextItem cur, nxt;
    prepare_item(p, BS, scan, claim.w, hkv, cur);
    for (long long k = 0;; ++k) {
        const int s = cur.s, kvh = cur.head, part = cur.part;
        const int slot = static_cast<int>(k % kGqaItemSlots);
        if (!mbar_wait_bounded(&iempty[slot], static_cast<uint32_t>((k / kGqaItemSlots) & 1) ^ 1u)) {
            ok = false;
            break;
        }
        if (s < 0) {
            if (lane == 0) {
                items[slot].end = 1;
                mbar_arrive(&ifull[slot]);
            }
            __syncwarp();
            break;
        }
        const SeqSpan sp = cur.sp;
        const int blk_lo = cur.blk_lo;
        const int nb = cur.nb;
        const int ntiles = (nb + C::kBpt - 1) / C::kBpt;
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
            it.t_first = static_cast<int>(t);
            it.end = 0;
            items[slot] = it;
            if (nb > 0) {
                mbar_arrive_expect_tx(&ifull[slot], 2 * G * 128);
                char *qs = qbuf + slot * C::kOpBytes;
                const int y = s * p.num_heads + kvh * G;
                tma_load_2d(qs, tmq, 0, y, &ifull[slot]);
                tma_load_2d(qs + 16 * 128, tmq, 64, y, &ifull[slot]);
            } else {
                mbar_arrive(&ifull[slot]);
            }
        }
        store_table(p, cur, tbl);
        __syncwarp();
        bool have_next = false;
        for (int ti = 0; ti < ntiles; ++ti, ++t) {
            const int stage = static_cast<int>(t % S);
            // the K half is free (S of tile t - S finished, the softmax warps
            // read its block mask) and the V producer took tile t - S's record
            if (!mbar_wait_bounded(&kempty[stage], ((t / S) & 1u) ^ 1u) ||
                !mbar_wait_bounded(&zfree[stage], ((t / S) & 1u) ^ 1u)) {
                ok = false;
                break;
            }
            // lane j issues the K copy of block j of the tile and leaves its
            // tile index for the V producer
            const int bj = ti * C::kBpt + lane;
            const bool mine = lane < C::kBpt && bj < nb && tbl[bj] >= 0;
            const uint32_t mask = __ballot_sync(0xffffffffu, mine);
            const int z = mine ? kv_tile(p, s, kvh, tbl[bj]) : 0;
            // a contiguous cache holds a whole tile's blocks in consecutive
            // tiles: one copy brings all of them
            const bool wide = p.contiguous && mask == C::kFullMask;
            if (lane < C::kBpt)
                zid[stage * kGqaMaxBpt + lane] = z;
            if (lane == 0) {
                meta[stage] = mask;
                zmask[stage] = mask;
                if (mask)
                    mbar_arrive_expect_tx(&kfull[stage], __popc(mask) * C::kBlockBytes);
                else
                    mbar_arrive(&kfull[stage]);
            }
            __syncwarp();
            if (wide ? lane == 0 : mine)
                tma_load_5d(stage_buf + static_cast<size_t>(stage) * 2 * C::kTile + lane * C::kBlockBytes,
                            wide ? tmkw : tmk, z, &kfull[stage], policy);
            if (lane == 0)
                mbar_arrive(&zfull[stage]);
            __syncwarp();
            if (ti == max(0, ntiles - kGqaNearTiles)) {  // the next item, while copies are in flight
                claim.next(p);
                prepare_item(p, BS, scan, claim.w, hkv, nxt);
                have_next = true;
            }
        }
        if (!ok)
            break;
        if (!have_next) {
            claim.next(p);
            prepare_item(p, BS, scan, claim.w, hkv, nxt);
        }
        cur = nxt;
    }
    // no more tiles for the V producer (after a failed wait too, so that it
    // stops without waiting out its own limit)
    if (lane == 0) {
        const int stage = static_cast<int>(t % S);
        if (!mbar_wait_bounded(&zfree[stage], ((t / S) & 1u) ^ 1u))
            ok = false;
        zmask[stage] = kGqaEndRecord;
        mbar_arrive(&zfull[stage]);
    }
    if (!ok && lane == 0) {
        // a wait gave up: flag it, then wait (bounded) for our copies in flight
        if (p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
        const uint32_t first = t > static_cast<uint32_t>(S) ? t - S : 0;
        for (uint32_t u = first; u < t; ++u)
            (void)mbar_wait_bounded(&kfull[u % S], (u / S) & 1u);
    }
    claim.finish(p);
    __syncwarp();
}

// The V producer (warp 6): for each tile, in order, the K producer's record
// (valid-block mask and tile indices), handed back as soon as it is read,
// then the V copies into the V half of the tile's stage once P V of tile
// t - S finished.
template <typename T, int BS, int G>
__device__ inline void gqa_vproducer(const DecodeParams &p, const CUtensorMap *tmv, const CUtensorMap *tmvw, char *smem,
                                     const GqaLayout &L) {
    using C = GqaCfg<T, BS, G>;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    uint64_t *vfull = reinterpret_cast<uint64_t *>(smem + L.vfull);
    uint64_t *vempty = reinterpret_cast<uint64_t *>(smem + L.vempty);
    uint64_t *zfull = reinterpret_cast<uint64_t *>(smem + L.zfull);
    uint64_t *zfree = reinterpret_cast<uint64_t *>(smem + L.zfree);
    const uint32_t *zmask = reinterpret_cast<const uint32_t *>(smem + L.zmask);
    const int32_t *zid = reinterpret_cast<const int32_t *>(smem + L.zid);
    char *stage_buf = smem + L.stages;
    const uint64_t policy = policy_evict_first();
    if (lane == 0)
        prefetch_tensormap(tmv);
    bool ok = true;
    uint32_t t = 0;
    for (;; ++t) {
        const int stage = static_cast<int>(t % S);
        if (!mbar_wait_bounded(&zfull[stage], (t / S) & 1u)) {
            ok = false;
            break;
        }
        const uint32_t mask = zmask[stage];
        if (mask == kGqaEndRecord)
            break;
        const int z = lane < C::kBpt ? zid[stage * kGqaMaxBpt + lane] : 0;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&zfree[stage]);  // the record is in registers
        if (!mbar_wait_bounded(&vempty[stage], ((t / S) & 1u) ^ 1u)) {
            ok = false;
            break;
        }
        if (lane == 0) {
            if (mask)
                mbar_arrive_expect_tx(&vfull[stage], __popc(mask) * C::kBlockBytes);
            else
                mbar_arrive(&vfull[stage]);
        }
        __syncwarp();
        const bool wide = p.contiguous && mask == C::kFullMask;
        if (wide ? lane == 0 : ((mask >> lane) & 1u) != 0)
            tma_load_5d(stage_buf + static_cast<size_t>(stage) * 2 * C::kTile + C::kTile + lane * C::kBlockBytes,
                        wide ? tmvw : tmv, z, &vfull[stage], policy);
        __syncwarp();
    }
    if (!ok && lane == 0) {
        if (p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
        const uint32_t first = t > static_cast<uint32_t>(S) ? t - S : 0;
        for (uint32_t u = first; u < t; ++u)
            (void)mbar_wait_bounded(&vfull[u % S], (u / S) & 1u);
    }
    __syncwarp();
}

// The single MMA-issuing thread (lane 0 of warp 1).  Tile g's S = K . Q^T is
// issued before tile g-1's P V, so the softmax of tile g overlaps the P V of
// tile g-1.
template <typename T, int BS, int G>
__device__ inline bool gqa_mma(const DecodeParams &p, char *smem, const GqaLayout &L, uint32_t tmem) {
    using C = GqaCfg<T, BS, G>;
    const int S = p.stages;
    uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + L.kfull);
    uint64_t *vfull = reinterpret_cast<uint64_t *>(smem + L.vfull);
    uint64_t *kempty = reinterpret_cast<uint64_t *>(smem + L.kempty);
    uint64_t *vempty = reinterpret_cast<uint64_t *>(smem + L.vempty);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint64_t *sfull = reinterpret_cast<uint64_t *>(smem + L.sfull);
    uint64_t *sfree = reinterpret_cast<uint64_t *>(smem + L.sfree);
    uint64_t *pfull = reinterpret_cast<uint64_t *>(smem + L.pfull);
    uint64_t *ofull = reinterpret_cast<uint64_t *>(smem + L.ofull);
    uint64_t *ofree = reinterpret_cast<uint64_t *>(smem + L.ofree);
    const MhaItem *items = reinterpret_cast<const MhaItem *>(smem + L.items);
    const char *qbuf = smem + L.qbuf;
    const char *pbuf = smem + L.pbuf;
    const char *stage_buf = smem + L.stages;
    constexpr uint32_t kIdQK = idesc_f16<T>(128, 16, 0, 0);
    constexpr uint32_t kIdPV = idesc_f16<T>(128, 16, 1, 0);

    // P V of a tile whose S was issued earlier: one accumulator per quarter of
    // the tile's tokens (the softmax warp that owns those tokens scales them).
    auto pv = [&](uint32_t gp, uint32_t tp) -> bool {
        const int b = static_cast<int>(gp & 1u);
        const uint32_t use = (gp >> 1) & 1u;
        const int stage_p = static_cast<int>(tp % S);
        if (!mbar_wait_bounded(&pfull[b], use) || !mbar_wait_bounded(&ofree[b], use ^ 1u) ||
            !mbar_wait_bounded(&vfull[stage_p], (tp / S) & 1u))
            return false;
        tc_fence_after();
        const char *vt = stage_buf + static_cast<size_t>(stage_p) * 2 * C::kTile + C::kTile;
        const char *pb = pbuf + b * C::kOpBytes;
#pragma unroll
        for (int w = 0; w < kGqaSmWarps; ++w) {
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int t0 = 32 * w + 16 * kk;  // first token of this K step
                // V^T, MN-major: head_dim halves C::kHalfBytes apart, 8-token groups
                // C::kGroupBytes apart (read either way round, every address stays
                // inside this tile)
                const uint64_t ad = sdesc(vt + (t0 >> 3) * C::kGroupBytes, C::kHalfBytes, C::kGroupBytes);
                const uint64_t bd = sdesc(pb + (t0 >> 6) * 16 * 128 + (t0 & 63) * 2, 16, 1024);
                tc_mma(tmem + 32 + b * 64 + w * 16, ad, bd, kIdPV, kk > 0);
            }
        }
        tc_commit(&ofull[b]);
        tc_commit(&vempty[stage_p]);  // the V half is free once P V finishes
        return true;
    };

    uint32_t g = 0;  // tiles whose S has been issued (S / P / O buffer = g & 1)
    bool have_prev = false;
    uint32_t prev_t = 0;
    for (int k = 0;; ++k) {
        const int slot = k % kGqaItemSlots;
        if (!mbar_wait_bounded(&ifull[slot], static_cast<uint32_t>(k / kGqaItemSlots) & 1u))
            return false;
        const MhaItem it = items[slot];
        if (it.end)
            break;
        const int ntiles = (it.nb + C::kBpt - 1) / C::kBpt;
        if (ntiles == 0) {
            mbar_arrive(&iempty[slot]);
            continue;
        }
        const char *qs = qbuf + slot * C::kOpBytes;
        for (int ti = 0; ti < ntiles; ++ti, ++g) {
            const uint32_t t = static_cast<uint32_t>(it.t_first + ti);
            const int stage = static_cast<int>(t % S);
            const int b = static_cast<int>(g & 1u);
            const uint32_t use = (g >> 1) & 1u;
            if (!mbar_wait_bounded(&kfull[stage], (t / S) & 1u) || !mbar_wait_bounded(&sfree[b], use ^ 1u))
                return false;
            tc_fence_after();
            const char *kt = stage_buf + static_cast<size_t>(stage) * 2 * C::kTile;
            // S = K . Q^T: A = K tile (K-major), B = Q (K-major); 8 steps of 16 along head_dim
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = sdesc(kt + (kk >> 2) * C::kHalfBytes + (kk & 3) * 32, 16, C::kGroupBytes);
                const uint64_t bd = sdesc(qs + (kk >> 2) * 16 * 128 + (kk & 3) * 32, 16, 1024);
                tc_mma(tmem + b * 16, ad, bd, kIdQK, kk > 0);
            }
            tc_commit(&sfull[b]);
            tc_commit(&kempty[stage]);  // the K half: once these MMAs finish (and the softmax warps read the mask)
            if (ti == ntiles - 1)
                tc_commit(&iempty[slot]);  // the query rows are free once these MMAs finish
            if (have_prev && !pv(g - 1, prev_t))
                return false;
            have_prev = true;
            prev_t = t;
        }
    }
    if (have_prev && !pv(g - 1, prev_t))
        return false;
    return true;
}

// Exchange N floats between the four softmax warps, double-buffered.
template <int N>
__device__ inline bool gqa_exchange(const float *v, float *all, float *xbuf, uint64_t *xfull, uint32_t &xc,
                                    int quarter, int lane) {
    const int b = static_cast<int>(xc & 1u);
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            xbuf[(b * kGqaSmWarps + quarter) * 16 + i] = v[i];
    }
    __syncwarp();
    if (lane == 0)
        mbar_arrive(&xfull[b]);
    if (!mbar_wait_bounded(&xfull[b], (xc >> 1) & 1u))
        return false;
#pragma unroll
    for (int w = 0; w < kGqaSmWarps; ++w)
#pragma unroll
        for (int i = 0; i < N; ++i)
            all[w * N + i] = xbuf[(b * kGqaSmWarps + w) * 16 + i];
    ++xc;
    return true;
}

// Softmax and epilogue warps.
template <typename T, int BS, int G>
__device__ inline bool gqa_softmax(const DecodeParams &p, char *smem, const GqaLayout &L, uint32_t tmem) {
    using C = GqaCfg<T, BS, G>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;            // tensor-memory lane quarter of this warp
    const int row = quarter * 32 + lane;     // tile token (S row) and head_dim index (O^T row)
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int S = p.stages;
    uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + L.kfull);
    uint64_t *vfull = reinterpret_cast<uint64_t *>(smem + L.vfull);
    uint64_t *kempty = reinterpret_cast<uint64_t *>(smem + L.kempty);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint64_t *sfull = reinterpret_cast<uint64_t *>(smem + L.sfull);
    uint64_t *sfree = reinterpret_cast<uint64_t *>(smem + L.sfree);
    uint64_t *pfull = reinterpret_cast<uint64_t *>(smem + L.pfull);
    uint64_t *ofull = reinterpret_cast<uint64_t *>(smem + L.ofull);
    uint64_t *ofree = reinterpret_cast<uint64_t *>(smem + L.ofree);
    uint64_t *xfull = reinterpret_cast<uint64_t *>(smem + L.xfull);
    const uint32_t *meta = reinterpret_cast<const uint32_t *>(smem + L.meta);
    const MhaItem *items = reinterpret_cast<const MhaItem *>(smem + L.items);
    float *xbuf = reinterpret_cast<float *>(smem + L.xbuf);
    // per-tile rescale factors [tile & 3][quarter][8]: a warp scoring tile x
    // implies every warp finished the epilogue of tile x - 4 (the P V of x - 2
    // waited for it before the S of x was issued), so four slots never collide
    float *abuf = reinterpret_cast<float *>(smem + L.abuf);
    char *pbuf = smem + L.pbuf;
    char *stage_buf = smem + L.stages;

    // P^T element (n, token) inside the 128-byte-swizzled K-major operand
    const int pbox = row >> 6;
    const int pchunk = (row & 63) >> 3;
    const int psub = (row & 7) * 2;

    // softmax state of the item being scored (per warp: uniform over lanes)
    float m_run[G], l_run[G];
    // epilogue state of the item being accumulated: one running output per quarter
    float o_run[kGqaSmWarps][G];
#pragma unroll
    for (int w = 0; w < kGqaSmWarps; ++w)
#pragma unroll
        for (int h = 0; h < G; ++h)
            o_run[w][h] = 0.f;
    // the tile whose epilogue is pending, and the finished item it may close
    bool pend = false, pend_last = false;
    uint32_t pend_g = 0;
    MhaItem pend_it = {};
    float fin_m[G], fin_l[G];

    uint32_t g = 0, xc = 0;

    // epilogue of tile gp; closes its item when it is the item's last tile
    auto epilogue = [&](uint32_t gp, bool last, const MhaItem &it) -> bool {
        const int b = static_cast<int>(gp & 1u);
        const uint32_t use = (gp >> 1) & 1u;
        if (!mbar_wait_bounded(&pfull[b], use) || !mbar_wait_bounded(&ofull[b], use))
            return false;
        tc_fence_after();
#pragma unroll
        for (int w = 0; w < kGqaSmWarps; ++w) {
            float ov[2 * G];
            tmem_ld<2 * G>(tl + 32 + b * 64 + w * 16, ov);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < G; ++h)
                o_run[w][h] = fmaf(o_run[w][h], abuf[((gp & 3u) * kGqaSmWarps + w) * 8 + h], ov[h] + ov[G + h]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&ofree[b]);
        if (!last)
            return true;
        // merge the four quarters: M = max m_w, out = sum o_w 2^(m_w - M) / sum l_w 2^(m_w - M)
        float ml[2 * G], all[kGqaSmWarps * 2 * G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float x = fin_l[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                x += __shfl_xor_sync(0xffffffffu, x, o);
            ml[h] = fin_m[h];
            ml[G + h] = x;
        }
        if (!gqa_exchange<2 * G>(ml, all, xbuf, xfull, xc, quarter, lane))
            return false;
        const long long row0 = static_cast<long long>(it.s) * p.num_heads + static_cast<long long>(it.kvh) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kGqaSmWarps; ++w)
                M = fmaxf(M, all[w * 2 * G + h]);
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kGqaSmWarps; ++w) {
                    const float sc = fast_exp2(all[w * 2 * G + h] - M);
                    num = fmaf(o_run[w][h], sc, num);
                    den = fmaf(all[w * 2 * G + G + h], sc, den);
                }
            }
            if (it.nparts == 1 && !p.force_partial) {
                store_out(p.out, p.out_dtype, (row0 + h) * C::kD + row, den > 0.f ? num / den : 0.f);
            } else {
                const long long pr = (row0 + h) * p.max_parts + it.part;
                p.part_acc[pr * C::kD + row] = num;
                if (row == 0) {
                    p.part_ml[pr * 2] = M;
                    p.part_ml[pr * 2 + 1] = den;
                }
            }
#pragma unroll
            for (int w = 0; w < kGqaSmWarps; ++w)
                o_run[w][h] = 0.f;
        }
        return true;
    };

    for (int k = 0;; ++k) {
        const int slot = k % kGqaItemSlots;
        if (!mbar_wait_bounded(&ifull[slot], static_cast<uint32_t>(k / kGqaItemSlots) & 1u))
            return false;
        const MhaItem it = items[slot];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&iempty[slot]);
        if (it.end)
            break;
        const int ntiles = (it.nb + C::kBpt - 1) / C::kBpt;
        if (ntiles == 0) {  // no attended token: zeros (or an empty partial), nothing to accumulate
            const long long row0 = static_cast<long long>(it.s) * p.num_heads + static_cast<long long>(it.kvh) * G;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if (!p.force_partial) {
                    store_out(p.out, p.out_dtype, (row0 + h) * C::kD + row, 0.f);
                } else {
                    const long long pr = (row0 + h) * p.max_parts + it.part;
                    p.part_acc[pr * C::kD + row] = 0.f;
                    if (row == 0) {
                        p.part_ml[pr * 2] = -INFINITY;
                        p.part_ml[pr * 2 + 1] = 0.f;
                    }
                }
            }
            continue;
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
            m_run[h] = -INFINITY, l_run[h] = 0.f;

        for (int ti = 0; ti < ntiles; ++ti, ++g) {
            const uint32_t t = static_cast<uint32_t>(it.t_first + ti);
            const int stage = static_cast<int>(t % S);
            const int b = static_cast<int>(g & 1u);
            const uint32_t use = (g >> 1) & 1u;
            if (!mbar_wait_bounded(&kfull[stage], (t / S) & 1u) || !mbar_wait_bounded(&sfull[b], use))
                return false;
            tc_fence_after();
            float sc[G];
            tmem_ld<G>(tl + b * 16, sc);
            const uint32_t mask = meta[stage];
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            // S and the tile's block mask are read: S buffer b and the K half
            // of the stage may be refilled
            if (lane == 0) {
                mbar_arrive(&sfree[b]);
                mbar_arrive(&kempty[stage]);
            }

            const int j = row / BS;
            const int tok = (it.blk_lo + ti * C::kBpt + j) * BS + (row % BS);
            const bool valid = ((mask >> j) & 1u) && tok >= it.tok_lo && tok < it.tok_hi;
            char *pb = pbuf + b * C::kOpBytes + pbox * 16 * 128;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float x = valid ? sc[h] * p.scale_log2 : -INFINITY;
                float mt = x;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                const float mn = fmaxf(m_run[h], mt);
                const float alpha = (mn == -INFINITY) ? 1.f : fast_exp2(m_run[h] - mn);
                m_run[h] = mn;
                const float pw = valid ? fast_exp2(x - mn) : 0.f;
                l_run[h] = l_run[h] * alpha + pw;
                if (lane == 0)
                    abuf[((g & 3u) * kGqaSmWarps + quarter) * 8 + h] = alpha;
                const uint16_t hi = to_bits16<T>(pw);
                const uint16_t lo = to_bits16<T>(pw - from_bits16<T>(hi));
                *reinterpret_cast<uint16_t *>(pb + h * 128 + ((pchunk ^ (h & 7)) << 4) + psub) = hi;
                *reinterpret_cast<uint16_t *>(pb + (G + h) * 128 + ((pchunk ^ ((G + h) & 7)) << 4) + psub) = lo;
            }
            // p = 0 for an invalid token; its V row must hold no NaN / Inf, so
            // it is zeroed once the tile's V has landed
            if (__any_sync(0xffffffffu, !valid) && !mbar_wait_bounded(&vfull[stage], (t / S) & 1u))
                return false;
            if (!valid) {
                char *vt = stage_buf + static_cast<size_t>(stage) * 2 * C::kTile + C::kTile;
#pragma unroll
                for (int bx = 0; bx < 2; ++bx) {
                    uint4 *dst = reinterpret_cast<uint4 *>(vt + (row >> 3) * C::kGroupBytes + bx * C::kHalfBytes +
                                                           (row & 7) * 128);
                    // chunk order rotated by the row: the lanes of a store cover
                    // eight chunk positions, i.e. all 32 banks (rows 128 bytes
                    // apart would otherwise all hit the same four)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        dst[(c + row) & 7] = make_uint4(0, 0, 0, 0);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&pfull[b]);

            if (pend && !epilogue(pend_g, pend_last, pend_it))
                return false;
            pend = true;
            pend_g = g;
            pend_last = (ti == ntiles - 1);
            pend_it = it;
            if (pend_last) {
#pragma unroll
                for (int h = 0; h < G; ++h)
                    fin_m[h] = m_run[h], fin_l[h] = l_run[h];
            }
        }
    }
    if (pend && !epilogue(pend_g, pend_last, pend_it))
        return false;
    return true;
}

template <typename T, int BS, int G>
__global__ void __launch_bounds__(kGqaThreads, 1)
    pa_decode_gqa_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq,
                         const __grid_constant__ CUtensorMap tmkw, const __grid_constant__ CUtensorMap tmvw) {
    // the next kernel on the stream may be launched now (it waits for this
    // grid); this one waits for the kernel before it
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using C = GqaCfg<T, BS, G>;
    const GqaLayout L = gqa_smem_layout(p.stages);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.kfull) + i, 1);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.vfull) + i, 1);
            // the S commit and the softmax warps (block mask read)
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.kempty) + i, 1 + kGqaSmWarps);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.vempty) + i, 1);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.zfull) + i, 1);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.zfree) + i, 1);
        }
        uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
        uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
        for (int i = 0; i < kGqaItemSlots; ++i) {
            mbar_init(&ifull[i], 1);
            mbar_init(&iempty[i], kGqaSmWarps + 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.sfull) + i, 1);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.sfree) + i, kGqaSmWarps);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.pfull) + i, kGqaSmWarps);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.ofull) + i, 1);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.ofree) + i, kGqaSmWarps);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.xfull) + i, kGqaSmWarps);
        }
        mbar_init(reinterpret_cast<uint64_t *>(smem + L.done), kGqaSmWarps);
        mbar_init(reinterpret_cast<uint64_t *>(smem + L.fin), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(reinterpret_cast<uint32_t *>(smem + L.tmem), kTmemCols);
        tmem_relinquish();
    }
    // zero the query and P operand buffers: rows beyond the G heads (and the
    // unused lo/hi rows) stay zero for the whole kernel
    {
        uint4 *z = reinterpret_cast<uint4 *>(smem + L.qbuf);
        const int n = (kGqaItemSlots * C::kOpBytes + 2 * C::kOpBytes) / 16;
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            z[i] = make_uint4(0, 0, 0, 0);
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L.tmem);

    if (warp == 0) {
        gqa_producer<T, BS, G>(p, &tmk, &tmkw, &tmq, smem, L);
    } else if (warp == 6) {
        gqa_vproducer<T, BS, G>(p, &tmv, &tmvw, smem, L);
    } else if (warp == 1) {
        bool ok = true;
        if ((threadIdx.x & 31) == 0) {
            ok = gqa_mma<T, BS, G>(p, smem, L, tmem);
            // every MMA this thread issued has finished before tensor memory goes
            tc_commit(reinterpret_cast<uint64_t *>(smem + L.fin));
            (void)mbar_wait_bounded(reinterpret_cast<uint64_t *>(smem + L.fin), 0);
            if (!ok && p.err)
                atomicOr(p.err, PA_DEVERR_TIMEOUT);
            // the softmax warps are done reading tensor memory
            (void)mbar_wait_bounded(reinterpret_cast<uint64_t *>(smem + L.done), 0);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    } else {
        const bool ok = gqa_softmax<T, BS, G>(p, smem, L, tmem);
        if (!ok && (threadIdx.x & 31) == 0 && p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
        tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0)
            mbar_arrive(reinterpret_cast<uint64_t *>(smem + L.done));
    }
    __syncthreads();
    release_claims(p);
}

}  // namespace pa
