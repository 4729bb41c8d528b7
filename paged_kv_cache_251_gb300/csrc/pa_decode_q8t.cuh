// Paged decode attention over an E4M3 KV cache on the 5th-generation tensor
// cores: tcgen05.mma kind::f8f6f4 multiplies the pages' codes as they land,
// accumulators in tensor memory.
//
// What it computes is the 8-bit-cache decode (pa_quant.cuh): for token t with
// key codes c_t, value codes c'_t and row scales sk_t, sv_t,
//   x_t = scale * sk_t * <q, c_t>,  out = sum_t e^(x_t - m) sv_t c'_t / sum_t e^(x_t - m),
// over the attended tokens reached through the block table
// ("PagedAttention — 把 KV cache 当虚拟内存页来管理", 案例 2; "KV Cache与长上下文管理",
// KV-cache quantisation), long contexts split into partitions merged by the
// log-sum-exp reduce.
//
// Items are (sequence, 4 consecutive kv heads, partition).  A block's pages of
// those heads are adjacent in the pool, so one 3-D TMA copy (128-byte swizzle)
// brings the block's 4 x block_size code rows of 128 bytes, and a second,
// unswizzled copy the pages' row scales.  128 code rows (2 blocks at block
// size 16, 1 at 32), ordered [block][kv head][row], form a tile: the MMA's
// M = 128.
//  - S = K . Q^T (N = 4 kv heads x 16 columns, K = head_dim).  The columns of
//    kv head h are (query g, term c) for its G query heads: the query row,
//    scaled by a power of two, written as three E4M3 terms q0 + q1/16 + q2/256
//    (exact for fp16 and bf16 queries).  A tile row takes the columns of its
//    own kv head; the others are computed and ignored.
//  - softmax: one thread per tile row; the rows of one kv head form a segment
//    of the warp (16 lanes at block size 16, 32 at 32) with its own running
//    max and denominator per query.  The thread applies sk, and writes its
//    weight p * sv (times a power of two per segment and tile) as three E4M3
//    terms into P^T, in its own kv head's columns only; every other entry of P
//    stays zero, so a product over rows of several kv heads keeps them apart.
//  - O^T = V^T . P per warp quarter of 32 tile rows (M = head_dim = 128,
//    N = the quarter's kv heads x 16 columns, K = 32 rows): V^T is the V code
//    tile read MN-major.
// Warps: 0 producer; 1 tensor-memory owner and issuer of S; 2..5 softmax;
// 6..9 epilogue (one accumulator per quarter, rescaled per tile, merged per
// item); 10 issuer of P V; 11 query converter.
// Every wait is bounded (PA_DEVERR_TIMEOUT); tensor memory is freed on every
// path; bad table entries are never dereferenced (PA_DEVERR_BAD_BLOCK).
#pragma once

#include "pa_decode_gqa.cuh"
#include "pa_quant.cuh"

namespace pa {

constexpr int kQ8tHeads = 4;   // kv heads per item
constexpr int kQ8tCols = 16;   // S / P columns per kv head: G queries x 3 terms, zero padded
constexpr int kQ8tTerms = 3;   // E4M3 terms of a query element or of a softmax weight
constexpr int kQ8tThreads = 12 * 32;  // producer, S issuer, 4 softmax, 4 epilogue, P V issuer, query converter
constexpr int kQ8tItemSlots = 4;
constexpr int kQ8tStages = 5;
constexpr int kQ8tMaxG = 4;
constexpr int kQ8tNearTiles = 4;  // an item's tiles still to issue when the next item is claimed
constexpr int kQ8tTile = kTileTokens * 128;            // codes of one operand (16 KB)
constexpr int kQ8tScales = kTileTokens * 4;            // row scales of one operand
constexpr int kQ8tStage = 2 * kQ8tTile + 2 * kQ8tScales;  // K codes, V codes, K scales, V scales
constexpr int kQ8tOp = kQ8tHeads * kQ8tCols * 128;     // Q or P operand: 64 rows x 128 bytes

struct Q8tItem {
    int s, kvh0, part, nparts;  // sequence, first kv head, partition, partitions of the sequence
    int nb;                     // blocks of the item (0: empty sequence)
    int tok_lo, tok_hi;         // attended tokens of the item: [tok_lo, tok_hi)
    int blk_lo;                 // first logical block
    int t_first;                // pipeline tile counter of the first tile
    int end;                    // 1: no more items
    int pad0, pad1;
};

template <int BS, int G> struct Q8tCfg {
    static constexpr int kR = kQ8tHeads * BS;         // tile rows per block
    static constexpr int kBpt = kTileTokens / kR;     // blocks per tile
    static constexpr int kQH = 32 / BS;               // kv heads in one warp quarter's rows
    static constexpr int kNs = kQ8tHeads * kQ8tCols;  // S columns
    static constexpr int kNq = kQH * kQ8tCols;        // P V columns of one quarter
    static constexpr uint32_t kTmemO = 2 * kNs;       // S[2] at column 0, O[2][4 quarters] after
    static constexpr uint32_t kTmemCols = (2 * kNs + 8 * kNq) <= 256 ? 256 : 512;
    static_assert(BS == 16 || BS == 32, "block size");
    static_assert(G >= 1 && G <= kQ8tMaxG && G * kQ8tTerms <= kQ8tCols, "query group");
    static_assert(2 * kNs + 8 * kNq <= 512, "tensor memory");
    // first kv head (within the item) among the tile rows of warp quarter w
    __host__ __device__ static constexpr int first_head(int w) { return (32 * w % kR) / BS; }
};

struct Q8tLayout {
    uint32_t full, empty, ifull, iempty, wfull, pnear, sfull, sfree, pfull, afull, ofull, ofree, done, fin, fin2;
    uint32_t meta, items, witem, tmem, table, qf, fbuf, abuf, qbuf, pbuf, stages, total;
};

__host__ __device__ inline Q8tLayout q8t_smem_layout(int S) {
    Q8tLayout L;
    uint32_t off = 0;
    L.full = off;
    off += 8 * S;
    L.empty = off;
    off += 8 * S;
    L.ifull = off;
    off += 8 * kQ8tItemSlots;
    L.iempty = off;
    off += 8 * kQ8tItemSlots;
    L.wfull = off;
    off += 8 * kQ8tItemSlots;
    L.pnear = off;
    off += 8 * kQ8tItemSlots;
    L.sfull = off;
    off += 16;
    L.sfree = off;
    off += 16;
    L.pfull = off;
    off += 16;
    L.afull = off;
    off += 32;
    L.ofull = off;
    off += 16;
    L.ofree = off;
    off += 16;
    L.done = off;
    off += 8;
    L.fin = off;
    off += 8;
    L.fin2 = off;
    off += 8;
    L.meta = off;
    off += 4 * S;
    L.items = align_up(off, 16);
    off = L.items + sizeof(Q8tItem) * kQ8tItemSlots;
    L.witem = off;  // item index of each slot, from the query converter to the producer
    off += 8 * kQ8tItemSlots;
    L.tmem = off;
    off += 16;
    L.table = off;
    off += 4 * kMaxBpp;
    L.qf = off;  // score factor per (item slot, kv head, query)
    off += 4 * kQ8tItemSlots * kQ8tHeads * kQ8tMaxG;
    L.fbuf = align_up(off, 16);  // item-final softmax state: [tile & 3][quarter][16]
    off = L.fbuf + 4 * 4 * 16 * 4;
    L.abuf = off;  // per-tile factors: [tile & 3][quarter][16]
    off += 4 * 4 * 16 * 4;
    L.qbuf = align_up(off, 1024);
    off = L.qbuf + kQ8tItemSlots * kQ8tOp;
    L.pbuf = off;
    off += 2 * kQ8tOp;
    L.stages = align_up(off, 1024);
    off = L.stages + S * kQ8tStage;
    L.total = off + 1024;  // slack to align the dynamic shared memory base
    return L;
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B: fp32 accumulate,
// A/B major-ness (0 = K-major, 1 = MN-major), N and M.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, int a_mn_major, int b_mn_major) {
    return (1u << 4) | (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D (+)= A . B^T; Acc = false overwrites D.
template <bool Acc>
__device__ inline void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "n"(Acc ? 1 : 0)
        : "memory");
}

// Shared-memory descriptors are advanced by byte offsets: the start-address
// field holds address / 16 in its low 14 bits, and every operand of this
// kernel lies below 256 KB, so the addition never carries out of the field.
__device__ inline uint64_t desc_at(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

template <> __device__ inline void tmem_ld<32>(uint32_t taddr, float *v) {
    tmem_ld<16>(taddr, v);
    tmem_ld<16>(taddr + 16, v + 16);
}

__device__ inline void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar,
                                   uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ inline uint2 ld_nc_v2(const void *p) {
    uint2 r;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// Two floats -> two E4M3 codes (x0's in the low byte): nearest, ties to even,
// saturating at +-448.
__device__ inline uint32_t e4m3x2_rn(float x0, float x1) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3));
}
// Two E4M3 codes (low byte first) -> their exact values.
__device__ inline float2 e4m3x2_value(uint32_t c2) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(c2 & 0xffffu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}
// x0, x1 (|x| < 448) as three E4M3 terms each, x ~ t0 + t1 / 16 + t2 / 256:
// each term codes 16 times the error left by the ones before it (the
// differences are exact in fp32).  c[i] holds the two codes of term i.
__device__ inline void e4m3_split3(float x0, float x1, uint32_t *c) {
    c[0] = e4m3x2_rn(x0, x1);
    float2 v = e4m3x2_value(c[0]);
    const float r0 = (x0 - v.x) * 16.f, r1 = (x1 - v.y) * 16.f;
    c[1] = e4m3x2_rn(r0, r1);
    v = e4m3x2_value(c[1]);
    c[2] = e4m3x2_rn((r0 - v.x) * 16.f, (r1 - v.y) * 16.f);
}

// Byte offset of element (row n, k) of a K-major operand of 128-byte rows in
// 8-row groups of 1024 bytes, 128-byte swizzle (k = byte within the row).
__device__ inline uint32_t sw128_offset(int n, int k) {
    return static_cast<uint32_t>((n >> 3) * 1024 + (n & 7) * 128 + ((((k >> 4) ^ (n & 7)) << 4) | (k & 15)));
}

// Power-of-two factors for a positive magnitude a: up = 2^(134 - e) brings a
// into [128, 256) (e = a's biased exponent, clamped so both factors are
// normal floats), down = 1 / up.
__device__ inline void q8t_pow2(float a, float &up, float &down) {
    int e = (__float_as_int(a) >> 23) & 0xff;
    e = e < 8 ? 8 : (e > 254 ? 254 : e);
    up = __int_as_float((261 - e) << 23);
    down = __int_as_float((e - 7) << 23);
}

// ---------------------------------------------------------------------------

// The walk over a CTA's items: item w is (item w / groups of the common order
// (ItemScan), kv-head group w % groups).  The producer and the query converter
// each run one.
template <int BS> struct Q8tScan {
    ItemScan scan;

    struct Found {
        int s, part, len, start, kvh0;
    };
    __device__ Found find(const DecodeParams &p, long long w, bool) {
        const long long nquads = p.num_kv_heads / kQ8tHeads;
        Found r{-1, 0, 0, 0, static_cast<int>(w % nquads) * kQ8tHeads};
        r.s = scan.find(p, BS, w / nquads, r.part, r.len, r.start);
        return r;
    }
    // the item's span and blocks
    __device__ static int blocks(const DecodeParams &p, const Found &it, SeqSpan &sp, int &blk_lo) {
        sp = seq_span(it.len, p.max_len, p.window, BS, p.bpp, it.start);
        blk_lo = sp.b0 + it.part * p.bpp;
        return max(0, min(p.bpp, sp.nblk - it.part * p.bpp));
    }
};

// Producer (warp 0): item records, block-table slices and the K / V copies.
template <int BS, int G>
__device__ inline void q8t_producer(const DecodeParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                    const CUtensorMap *tsk, const CUtensorMap *tsv, char *smem, const Q8tLayout &L) {
    using C = Q8tCfg<BS, G>;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint32_t *meta = reinterpret_cast<uint32_t *>(smem + L.meta);
    Q8tItem *items = reinterpret_cast<Q8tItem *>(smem + L.items);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + L.table);
    char *stage_buf = smem + L.stages;
    const uint64_t policy = policy_evict_first();
    if (lane == 0) {
        prefetch_tensormap(tmk);
        prefetch_tensormap(tmv);
        prefetch_tensormap(tsk);
        prefetch_tensormap(tsv);
    }
    uint64_t *wfull = reinterpret_cast<uint64_t *>(smem + L.wfull);
    uint64_t *pnear = reinterpret_cast<uint64_t *>(smem + L.pnear);
    const long long *witem = reinterpret_cast<const long long *>(smem + L.witem);
    Q8tScan<BS> scan;
    uint32_t t = 0;
    bool ok = true;
    for (long long k = 0;; ++k) {
        const int slot = static_cast<int>(k % kQ8tItemSlots);
        // the item index comes from the query converter, which picks it
        if (!mbar_wait_bounded(&iempty[slot], static_cast<uint32_t>((k / kQ8tItemSlots) & 1) ^ 1u) ||
            !mbar_wait_bounded(&wfull[slot], static_cast<uint32_t>(k / kQ8tItemSlots) & 1u)) {
            ok = false;
            break;
        }
        const auto it0 = scan.find(p, witem[slot], true);
        const int s = it0.s, kvh0 = it0.kvh0;
        if (s < 0) {
            if (lane == 0) {
                items[slot].end = 1;
                mbar_arrive(&ifull[slot]);
            }
            __syncwarp();
            break;
        }
        SeqSpan sp;
        int blk_lo;
        const int nb = Q8tScan<BS>::blocks(p, it0, sp, blk_lo);
        const int ntiles = (nb + C::kBpt - 1) / C::kBpt;
        if (lane == 0) {
            Q8tItem it;
            it.s = s;
            it.kvh0 = kvh0;
            it.part = it0.part;
            it.nparts = sp.nparts;
            it.nb = nb;
            it.tok_lo = max(sp.start, blk_lo * BS);
            it.tok_hi = min(sp.end, (blk_lo + nb) * BS);
            it.blk_lo = blk_lo;
            it.t_first = static_cast<int>(t);
            it.end = 0;
            it.pad0 = it.pad1 = 0;
            items[slot] = it;
            mbar_arrive(&ifull[slot]);  // the query converter arrives for the operand
            if (ntiles <= kQ8tNearTiles)
                mbar_arrive(&pnear[slot]);  // the next item may be claimed
        }
        __syncwarp();
        const int32_t *row = p.block_tables + static_cast<long long>(s) * p.max_blocks_per_seq + blk_lo;
        for (int j = lane; j < nb; j += 32) {
            int pb = ld_nc_i32(row + j);
            if (pb < 0 || pb >= p.num_blocks) {
                pb = -1;
                if (p.err)
                    atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
            }
            tbl[j] = pb;
        }
        __syncwarp();
        for (int ti = 0; ti < ntiles; ++ti, ++t) {
            const int stage = static_cast<int>(t % S);
            if (!mbar_wait_bounded(&empty[stage], ((t / S) & 1u) ^ 1u)) {
                ok = false;
                break;
            }
            // lane j issues block j of the tile: code rows and scale rows of K and V
            const int bj = ti * C::kBpt + lane;
            const bool mine = lane < C::kBpt && bj < nb && tbl[bj] >= 0;
            const uint32_t mask = __ballot_sync(0xffffffffu, mine);
            if (lane == 0) {
                meta[stage] = mask;
                if (mask)
                    mbar_arrive_expect_tx(&full[stage], __popc(mask) * 2 * (C::kR * 128 + C::kR * 4));
                else
                    mbar_arrive(&full[stage]);
            }
            __syncwarp();
            if (mine) {
                char *st = stage_buf + static_cast<size_t>(stage) * kQ8tStage;
                const int z = tbl[bj] * p.num_kv_heads + kvh0;
                tma_load_3d(st + lane * C::kR * 128, tmk, 0, 0, z, &full[stage], policy);
                tma_load_3d(st + kQ8tTile + lane * C::kR * 128, tmv, 0, 0, z, &full[stage], policy);
                tma_load_3d(st + 2 * kQ8tTile + lane * C::kR * 4, tsk, 0, BS, z, &full[stage], policy);
                tma_load_3d(st + 2 * kQ8tTile + kQ8tScales + lane * C::kR * 4, tsv, 0, BS, z, &full[stage], policy);
            }
            if (lane == 0 && ti == ntiles - 1 - kQ8tNearTiles)
                mbar_arrive(&pnear[slot]);  // the next item may be claimed
            __syncwarp();
        }
        if (!ok)
            break;
    }
    if (!ok && lane == 0) {
        // a wait gave up: flag it, then wait (bounded) for our copies in flight
        if (p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
        const uint32_t first = t > static_cast<uint32_t>(S) ? t - S : 0;
        for (uint32_t u = first; u < t; ++u)
            (void)mbar_wait_bounded(&full[u % S], (u / S) & 1u);
    }
    __syncwarp();
}

// Query converter (warp 11): for each item, its 4 x G query rows (consecutive
// in q) as the B operand of S in the item's slot: row (kv head h, query g,
// term c) = h * 16 + 3 g + c, each query row scaled by a power of two (its
// score factor goes to qf).  It walks the same items as the producer and
// claims item k once the producer has kQ8tNearTiles tiles of item k - 1 left.
template <int BS, int G>
__device__ inline bool q8t_qconvert(const DecodeParams &p, char *smem, const Q8tLayout &L) {
    constexpr int kRows = kQ8tHeads * G;
    const int lane = threadIdx.x & 31;
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    float *qfs = reinterpret_cast<float *>(smem + L.qf);
    char *qbuf = smem + L.qbuf;
    const char *qg = static_cast<const char *>(p.q);
    uint64_t *wfull = reinterpret_cast<uint64_t *>(smem + L.wfull);
    uint64_t *pnear = reinterpret_cast<uint64_t *>(smem + L.pnear);
    long long *witem = reinterpret_cast<long long *>(smem + L.witem);
    Q8tScan<BS> scan;
    long long w = blockIdx.x;
    for (long long k = 0;; ++k) {
        const int slot = static_cast<int>(k % kQ8tItemSlots);
        if (!mbar_wait_bounded(&iempty[slot], static_cast<uint32_t>((k / kQ8tItemSlots) & 1) ^ 1u))
            return false;
        // the next item: the CTA's own first, then from the launch's shared
        // counter (each CTA takes the next unclaimed one when it has room;
        // the counter numbers them from gridDim.x up), else round-robin
        if (p.work && k > 0) {
            // item k is claimed once the producer has at most kQ8tNearTiles
            // tiles of item k - 1 left to issue: a CTA never holds a claimed
            // item it is far from starting, so the launch's last items go to
            // the CTAs that run out of work first
            const int ps = static_cast<int>((k - 1) % kQ8tItemSlots);
            if (!mbar_wait_bounded(&pnear[ps], static_cast<uint32_t>(((k - 1) / kQ8tItemSlots) & 1)))
                return false;
            unsigned int v = 0;
            if (lane == 0)
                v = gridDim.x + atomicAdd(p.work, 1u);
            w = __shfl_sync(0xffffffffu, v, 0);
        } else if (k > 0) {
            w += gridDim.x;
        }
        if (lane == 0) {
            witem[slot] = w;
            mbar_arrive(&wfull[slot]);
        }
        const auto it = scan.find(p, w, false);
        SeqSpan sp;
        int blk_lo;
        if (it.s >= 0 && Q8tScan<BS>::blocks(p, it, sp, blk_lo) > 0) {
            // lane l converts elements 4l .. 4l + 3 of every row; the rows proceed together
            const char *q0 =
                qg + (static_cast<long long>(it.s) * p.num_heads + static_cast<long long>(it.kvh0) * G) * 256;
            char *qs = qbuf + slot * kQ8tOp;
            float x[kRows][4], a[kRows];
            uint2 raw[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                raw[r] = ld_nc_v2(q0 + r * 256 + lane * 8);
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                if (p.q_dtype == PA_F16) {
                    const float2 u = __half22float2(*reinterpret_cast<const __half2 *>(&raw[r].x));
                    const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&raw[r].y));
                    x[r][0] = u.x, x[r][1] = u.y, x[r][2] = v.x, x[r][3] = v.y;
                } else {
                    x[r][0] = __uint_as_float(raw[r].x << 16), x[r][1] = __uint_as_float(raw[r].x & 0xffff0000u);
                    x[r][2] = __uint_as_float(raw[r].y << 16), x[r][3] = __uint_as_float(raw[r].y & 0xffff0000u);
                }
                a[r] = fmaxf(fmaxf(fabsf(x[r][0]), fabsf(x[r][1])), fmaxf(fabsf(x[r][2]), fabsf(x[r][3])));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int r = 0; r < kRows; ++r)
                    a[r] = fmaxf(a[r], __shfl_xor_sync(0xffffffffu, a[r], o));
            float my_qf = 0.f;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float up, down;
                q8t_pow2(a[r], up, down);
                my_qf = lane == r ? (a[r] > 0.f ? p.scale_log2 * down : 0.f) : my_qf;
                uint32_t lo[kQ8tTerms], hi[kQ8tTerms];
                e4m3_split3(x[r][0] * up, x[r][1] * up, lo);
                e4m3_split3(x[r][2] * up, x[r][3] * up, hi);
                const int h = r / G, g = r % G;
#pragma unroll
                for (int c = 0; c < kQ8tTerms; ++c) {
                    const int n = h * kQ8tCols + g * kQ8tTerms + c;
                    *reinterpret_cast<uint32_t *>(qs + sw128_offset(n, 4 * lane)) = (lo[c] & 0xffffu) | (hi[c] << 16);
                }
            }
            if (lane < kRows)
                qfs[slot * kQ8tHeads * kQ8tMaxG + lane] = my_qf;
            fence_async_smem();
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&ifull[slot]);
        if (it.s < 0)
            break;
    }
    if (p.work)
        __threadfence();  // the claims are complete before the CTA reports itself done
    return true;
}

// The two MMA-issuing threads.  S of every tile comes from lane 0 of warp 1,
// P V from lane 0 of warp 10: each waits while the other issues.
//
// S thread: S(g) needs its stage landed, S buffer g & 1 read by the softmax
// (tile g - 2) and P V of tile g - 2 complete: then the softmax, once it sees
// S(g), may overwrite P buffer g & 1 and the factor slot g & 3 (P V(g - 2)
// was issued after the epilogue of g - 4).
template <int BS, int G>
__device__ inline bool q8t_mma_s(const DecodeParams &p, char *smem, const Q8tLayout &L, uint32_t tmem) {
    using C = Q8tCfg<BS, G>;
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint64_t *sfull = reinterpret_cast<uint64_t *>(smem + L.sfull);
    uint64_t *sfree = reinterpret_cast<uint64_t *>(smem + L.sfree);
    uint64_t *ofull = reinterpret_cast<uint64_t *>(smem + L.ofull);
    const Q8tItem *items = reinterpret_cast<const Q8tItem *>(smem + L.items);
    constexpr uint32_t kIdS = idesc_e4m3(128, C::kNs, 0, 0);
    // K tiles and the query operand: K-major, 128-byte rows in 8-row groups of 1024 bytes
    const uint64_t dk = sdesc(smem + L.stages, 16, 1024);
    const uint64_t dq = sdesc(smem + L.qbuf, 16, 1024);
    uint32_t g = 0;  // tiles whose S has been issued (S / P / O buffer = g & 1)
    for (int k = 0;; ++k) {
        const int slot = k % kQ8tItemSlots;
        if (!mbar_wait_bounded(&ifull[slot], static_cast<uint32_t>(k / kQ8tItemSlots) & 1u))
            return false;
        const Q8tItem it = items[slot];
        if (it.end)
            break;
        const int ntiles = (it.nb + C::kBpt - 1) / C::kBpt;
        if (ntiles == 0) {
            mbar_arrive(&iempty[slot]);
            continue;
        }
        const uint64_t bq = desc_at(dq, static_cast<uint32_t>(slot) * kQ8tOp);
#pragma unroll 1
        for (int ti = 0; ti < ntiles; ++ti, ++g) {
            const uint32_t t = static_cast<uint32_t>(it.t_first + ti);
            const int stage = static_cast<int>(t % S);
            const int b = static_cast<int>(g & 1u);
            const uint32_t prev = ((g >> 1) & 1u) ^ 1u;  // phase parity of tile g - 2 on buffer b
            if (!mbar_wait_bounded(&full[stage], (t / S) & 1u) || !mbar_wait_bounded(&sfree[b], prev) ||
                !mbar_wait_bounded(&ofull[b], prev))
                return false;
            tc_fence_after();
            // S = K . Q^T: A = K codes, B = query terms; 4 steps of 32 along head_dim
            const uint64_t ak = desc_at(dk, static_cast<uint32_t>(stage) * kQ8tStage);
            const uint32_t dS = tmem + static_cast<uint32_t>(b) * C::kNs;
            tc_mma_f8<false>(dS, ak, bq, kIdS);
            tc_mma_f8<true>(dS, desc_at(ak, 32), desc_at(bq, 32), kIdS);
            tc_mma_f8<true>(dS, desc_at(ak, 64), desc_at(bq, 64), kIdS);
            tc_mma_f8<true>(dS, desc_at(ak, 96), desc_at(bq, 96), kIdS);
            tc_commit(&sfull[b]);
            if (ti == ntiles - 1)
                tc_commit(&iempty[slot]);  // the query operand is free once these MMAs finish
        }
    }
    return true;
}

// P V thread: P V(g) needs the softmax of tile g (its P and V rows) and the
// epilogue of tile g - 2 (accumulator buffer g & 1).  Its completion frees
// the stage: S(g) finished before the softmax of g could start.
template <int BS, int G>
__device__ inline bool q8t_mma_pv(const DecodeParams &p, char *smem, const Q8tLayout &L, uint32_t tmem) {
    using C = Q8tCfg<BS, G>;
    const int S = p.stages;
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint64_t *pfull = reinterpret_cast<uint64_t *>(smem + L.pfull);
    uint64_t *ofull = reinterpret_cast<uint64_t *>(smem + L.ofull);
    uint64_t *ofree = reinterpret_cast<uint64_t *>(smem + L.ofree);
    const Q8tItem *items = reinterpret_cast<const Q8tItem *>(smem + L.items);
    constexpr uint32_t kIdPV = idesc_e4m3(128, C::kNq, 1, 0);
    // V^T: MN-major, head_dim is one 128-byte swizzle row, 8-row groups 1024
    // bytes apart (both offsets 1024, whichever way they are read).  P: K-major.
    const uint64_t dv = sdesc(smem + L.stages + kQ8tTile, 1024, 1024);
    const uint64_t dp = sdesc(smem + L.pbuf, 16, 1024);
    uint32_t g = 0;
    for (int k = 0;; ++k) {
        const int slot = k % kQ8tItemSlots;
        if (!mbar_wait_bounded(&ifull[slot], static_cast<uint32_t>(k / kQ8tItemSlots) & 1u))
            return false;
        const Q8tItem it = items[slot];
        mbar_arrive(&iempty[slot]);
        if (it.end)
            break;
        const int ntiles = (it.nb + C::kBpt - 1) / C::kBpt;
#pragma unroll 1
        for (int ti = 0; ti < ntiles; ++ti, ++g) {
            const uint32_t t = static_cast<uint32_t>(it.t_first + ti);
            const int stage = static_cast<int>(t % S);
            const int b = static_cast<int>(g & 1u);
            const uint32_t use = (g >> 1) & 1u;
            if (!mbar_wait_bounded(&pfull[b], use) || !mbar_wait_bounded(&ofree[b], use ^ 1u))
                return false;
            tc_fence_after();
            // O^T = V^T . P, one accumulator per quarter of the tile's rows, over
            // the quarter's kv heads' columns of P
            const uint64_t av = desc_at(dv, static_cast<uint32_t>(stage) * kQ8tStage);
            const uint64_t bp = desc_at(dp, static_cast<uint32_t>(b) * kQ8tOp);
            const uint32_t dO = tmem + C::kTmemO + static_cast<uint32_t>(b) * 4 * C::kNq;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                tc_mma_f8<false>(dO + w * C::kNq, desc_at(av, w * 32 * 128),
                                 desc_at(bp, C::first_head(w) * kQ8tCols * 128 + w * 32), kIdPV);
            tc_commit(&ofull[b]);
            tc_commit(&empty[stage]);
        }
    }
    return true;
}

// Softmax warps (2..5): one thread per tile row.
template <int BS, int G>
__device__ inline bool q8t_softmax(const DecodeParams &p, char *smem, const Q8tLayout &L, uint32_t tmem) {
    using C = Q8tCfg<BS, G>;
    constexpr int kQH = C::kQH, kNq = C::kNq;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;             // tensor-memory lane quarter of this warp
    const int row = quarter * 32 + lane;      // tile row
    const int fh = C::first_head(quarter);    // first kv head among this warp's rows
    const int jb = row / C::kR;               // block of the tile holding the row
    const int hl = (row % C::kR) / BS;        // kv head of the row within the item
    const int hq = hl - fh;                   // its segment of the warp
    const int ri = row % BS;                  // row within the block (= lane within the segment)
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint64_t *sfull = reinterpret_cast<uint64_t *>(smem + L.sfull);
    uint64_t *sfree = reinterpret_cast<uint64_t *>(smem + L.sfree);
    uint64_t *pfull = reinterpret_cast<uint64_t *>(smem + L.pfull);
    uint64_t *afull = reinterpret_cast<uint64_t *>(smem + L.afull);
    const uint32_t *meta = reinterpret_cast<const uint32_t *>(smem + L.meta);
    const Q8tItem *items = reinterpret_cast<const Q8tItem *>(smem + L.items);
    const float *qfs = reinterpret_cast<const float *>(smem + L.qf);
    // per-tile factors [tile & 3][quarter][16]: entry 8 h + g is the rescale of
    // (segment h, query g), entry 8 h + 4 the power of two of segment h's P
    float *abuf = reinterpret_cast<float *>(smem + L.abuf);
    // an item's final softmax state, at its last tile: [tile & 3][quarter][16],
    // entry 8 h + g the running max, 8 h + 4 + g the denominator
    float *fbuf = reinterpret_cast<float *>(smem + L.fbuf);
    char *pbuf = smem + L.pbuf;
    char *stage_buf = smem + L.stages;

    float m_run[G], l_run[G], qf[G];
    uint32_t g = 0;
    for (int k = 0;; ++k) {
        const int slot = k % kQ8tItemSlots;
        if (!mbar_wait_bounded(&ifull[slot], static_cast<uint32_t>(k / kQ8tItemSlots) & 1u))
            return false;
        const Q8tItem it = items[slot];
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
            qf[gg] = qfs[slot * kQ8tHeads * kQ8tMaxG + hl * G + gg];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&iempty[slot]);
        if (it.end)
            break;
        const int ntiles = (it.nb + C::kBpt - 1) / C::kBpt;
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
            m_run[gg] = -INFINITY, l_run[gg] = 0.f;

#pragma unroll 1
        for (int ti = 0; ti < ntiles; ++ti, ++g) {
            const uint32_t t = static_cast<uint32_t>(it.t_first + ti);
            const int stage = static_cast<int>(t % S);
            const int b = static_cast<int>(g & 1u);
            const uint32_t use = (g >> 1) & 1u;
            if (!mbar_wait_bounded(&full[stage], (t / S) & 1u) || !mbar_wait_bounded(&sfull[b], use))
                return false;
            tc_fence_after();
            float sc[kNq];
            tmem_ld<kNq>(tl + b * C::kNs + fh * kQ8tCols, sc);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sfree[b]);

            char *st = stage_buf + static_cast<size_t>(stage) * kQ8tStage;
            const float ks = *reinterpret_cast<const float *>(st + 2 * kQ8tTile + 4 * row);
            const float vs = *reinterpret_cast<const float *>(st + 2 * kQ8tTile + kQ8tScales + 4 * row);
            const uint32_t mask = meta[stage];
            const int tok = (it.blk_lo + ti * C::kBpt + jb) * BS + ri;
            const bool valid = ((mask >> jb) & 1u) && tok >= it.tok_lo && tok < it.tok_hi;
            // this row's weights scaled into [0, 256) by a power of two per segment
            float vmax = valid ? vs : 0.f;
#pragma unroll
            for (int o = BS / 2; o > 0; o >>= 1)
                vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
            float up, down;
            q8t_pow2(vmax, up, down);
            const float vsu = vs * up;
            float *ab = abuf + ((g & 3u) * 4 + quarter) * 16 + hq * 8;
            float pw[G + (G & 1)];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                // this row's kv head's columns among the warp's (two heads at block size 16)
                float s0 = sc[gg * kQ8tTerms], s1 = sc[gg * kQ8tTerms + 1], s2 = sc[gg * kQ8tTerms + 2];
                if constexpr (kQH > 1) {
                    const float *sh = sc + kQ8tCols + gg * kQ8tTerms;
                    s0 = hq > 0 ? sh[0] : s0;
                    s1 = hq > 0 ? sh[1] : s1;
                    s2 = hq > 0 ? sh[2] : s2;
                }
                const float x = valid ? fmaf(s2, 0.00390625f, fmaf(s1, 0.0625f, s0)) * ks * qf[gg] : -INFINITY;
                float mt = x;
#pragma unroll
                for (int o = BS / 2; o > 0; o >>= 1)
                    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                const float mn = fmaxf(m_run[gg], mt);
                const float alpha = (mn == -INFINITY) ? 1.f : fast_exp2(m_run[gg] - mn);
                m_run[gg] = mn;
                const float e = valid ? fast_exp2(x - mn) : 0.f;
                l_run[gg] = l_run[gg] * alpha + e;
                pw[gg] = valid ? e * vsu : 0.f;
                if (ri == 0)
                    ab[gg] = alpha;
            }
            if (G & 1)
                pw[G] = 0.f;
            if (ri == 0)
                ab[4] = down;
            // P^T entries of this row in its kv head's columns (three terms each)
            char *pb = pbuf + b * kQ8tOp;
#pragma unroll
            for (int gp2 = 0; gp2 < (G + 1) / 2; ++gp2) {
                uint32_t c[kQ8tTerms];
                e4m3_split3(pw[2 * gp2], pw[2 * gp2 + 1], c);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int gg = 2 * gp2 + u;
                    if (gg < G) {
#pragma unroll
                        for (int cc = 0; cc < kQ8tTerms; ++cc) {
                            const int n = hl * kQ8tCols + gg * kQ8tTerms + cc;
                            pb[sw128_offset(n, row)] = static_cast<char>((c[cc] >> (8 * u)) & 0xffu);
                        }
                    }
                }
            }
            if (!valid) {  // its weight is 0; make sure its V codes are no NaN
                uint4 *dst = reinterpret_cast<uint4 *>(st + kQ8tTile + row * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_uint4(0, 0, 0, 0);
            }
            if (ti == ntiles - 1) {  // the item's final state for the epilogue warps' merge
                float *fb = fbuf + ((g & 3u) * 4 + quarter) * 16 + hq * 8;
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    float l = l_run[gg];
#pragma unroll
                    for (int o = BS / 2; o > 0; o >>= 1)
                        l += __shfl_xor_sync(0xffffffffu, l, o);
                    if (ri == 0) {
                        fb[gg] = m_run[gg];
                        fb[4 + gg] = l;
                    }
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&pfull[b]);
                mbar_arrive(&afull[g & 3u]);
            }
        }
    }
    return true;
}

// Epilogue warps (6..9): thread = head_dim row of O^T; one running output per
// (quarter, its kv head, query), rescaled per tile and merged per item.
template <int BS, int G>
__device__ inline bool q8t_epilogue(const DecodeParams &p, char *smem, const Q8tLayout &L, uint32_t tmem) {
    using C = Q8tCfg<BS, G>;
    constexpr int kQH = C::kQH, kNq = C::kNq;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // head_dim index
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint64_t *afull = reinterpret_cast<uint64_t *>(smem + L.afull);
    uint64_t *ofull = reinterpret_cast<uint64_t *>(smem + L.ofull);
    uint64_t *ofree = reinterpret_cast<uint64_t *>(smem + L.ofree);
    const Q8tItem *items = reinterpret_cast<const Q8tItem *>(smem + L.items);
    const float *abuf = reinterpret_cast<const float *>(smem + L.abuf);
    const float *fbuf = reinterpret_cast<const float *>(smem + L.fbuf);

    float o_run[4][kQH][G];
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
        for (int h = 0; h < kQH; ++h)
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
                o_run[w][h][gg] = 0.f;
    uint32_t g = 0;
    for (int k = 0;; ++k) {
        const int slot = k % kQ8tItemSlots;
        if (!mbar_wait_bounded(&ifull[slot], static_cast<uint32_t>(k / kQ8tItemSlots) & 1u))
            return false;
        const Q8tItem it = items[slot];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&iempty[slot]);
        if (it.end)
            break;
        const int ntiles = (it.nb + C::kBpt - 1) / C::kBpt;
        const long long row0 = static_cast<long long>(it.s) * p.num_heads + static_cast<long long>(it.kvh0) * G;
        if (ntiles == 0) {  // no attended token: zeros (or an empty partial)
#pragma unroll
            for (int r = 0; r < kQ8tHeads * G; ++r) {
                if (!p.force_partial) {
                    store_out(p.out, p.out_dtype, (row0 + r) * 128 + row, 0.f);
                } else {
                    const long long pr = (row0 + r) * p.max_parts + it.part;
                    p.part_acc[pr * 128 + row] = 0.f;
                    if (row == 0) {
                        p.part_ml[pr * 2] = -INFINITY;
                        p.part_ml[pr * 2 + 1] = 0.f;
                    }
                }
            }
            continue;
        }
#pragma unroll 1
        for (int ti = 0; ti < ntiles; ++ti, ++g) {
            const int b = static_cast<int>(g & 1u);
            const uint32_t use = (g >> 1) & 1u;
            // afull[g & 3]: every softmax warp's factors for tile g are in place.
            // A ring of 4, not the 2-deep pfull: the softmax warps may run two
            // tiles ahead of this warp (tile g + 2 needs only the epilogue of
            // g - 2), which would complete a 2-deep barrier's phase twice.
            // Tile g + 4 needs the epilogue of g, so 4 phases never alias.
            if (!mbar_wait_bounded(&afull[g & 3u], (g >> 2) & 1u) || !mbar_wait_bounded(&ofull[b], use))
                return false;
            tc_fence_after();
            const float *ab = abuf + (g & 3u) * 4 * 16;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
#pragma unroll
                for (int h = 0; h < kQH; ++h) {
                    float ov[kQ8tCols];
                    tmem_ld<kQ8tCols>(tl + C::kTmemO + (b * 4 + w) * kNq + h * kQ8tCols, ov);
                    tmem_wait_ld();
                    const float fv = ab[w * 16 + h * 8 + 4];
#pragma unroll
                    for (int gg = 0; gg < G; ++gg) {
                        const float *o3 = ov + gg * kQ8tTerms;
                        const float o = fmaf(o3[2], 0.00390625f, fmaf(o3[1], 0.0625f, o3[0]));
                        o_run[w][h][gg] = fmaf(o_run[w][h][gg], ab[w * 16 + h * 8 + gg], fv * o);
                    }
                }
            }
            tc_fence_before();
            if (ti < ntiles - 1) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ofree[b]);
                continue;
            }
            // merge the quarters holding each kv head:
            // out = sum_w o_w 2^(m_w - M) / sum_w l_w 2^(m_w - M), M = max_w m_w.
            // The item's final state in fbuf slot g & 3 is read before this warp
            // frees O buffer b: that release lets P V of tile g + 2 and then S
            // and the softmax of tile g + 4 go ahead, and the softmax rewrites
            // the slot if tile g + 4 ends an item.
            const float *fb = fbuf + (g & 3u) * 4 * 16;
#pragma unroll
            for (int h = 0; h < kQ8tHeads; ++h) {
#pragma unroll
                for (int gg = 0; gg < G; ++gg) {
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int hw = h - C::first_head(w);
                        if (hw >= 0 && hw < kQH)
                            M = fmaxf(M, fb[w * 16 + hw * 8 + gg]);
                    }
                    float num = 0.f, den = 0.f;
                    if (M != -INFINITY) {
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const int hw = h - C::first_head(w);
                            if (hw >= 0 && hw < kQH) {
                                const float sc = fast_exp2(fb[w * 16 + hw * 8 + gg] - M);
                                num = fmaf(o_run[w][hw][gg], sc, num);
                                den = fmaf(fb[w * 16 + hw * 8 + 4 + gg], sc, den);
                            }
                        }
                    }
                    const long long qrow = row0 + h * G + gg;
                    if (it.nparts == 1 && !p.force_partial) {
                        store_out(p.out, p.out_dtype, qrow * 128 + row, den > 0.f ? num / den : 0.f);
                    } else {
                        const long long pr = qrow * p.max_parts + it.part;
                        p.part_acc[pr * 128 + row] = num;
                        if (row == 0) {
                            p.part_ml[pr * 2] = M;
                            p.part_ml[pr * 2 + 1] = den;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ofree[b]);
#pragma unroll
            for (int w = 0; w < 4; ++w)
#pragma unroll
                for (int h = 0; h < kQH; ++h)
#pragma unroll
                    for (int gg = 0; gg < G; ++gg)
                        o_run[w][h][gg] = 0.f;
        }
    }
    return true;
}

template <int BS, int G>
__global__ void __launch_bounds__(kQ8tThreads, 1)
    pa_decode_q8t_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tsk,
                         const __grid_constant__ CUtensorMap tsv) {
    // the next kernel on the stream may be launched now (it waits for this
    // grid); this one waits for the kernel before it
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using C = Q8tCfg<BS, G>;
    if (p.stages < 2 || p.stages > 8 || p.num_kv_heads % kQ8tHeads != 0) {
        if (threadIdx.x == 0 && p.err)
            atomicOr(p.err, PA_DEVERR_BAD_LAUNCH);
        return;
    }
    const Q8tLayout L = q8t_smem_layout(p.stages);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
        uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
        uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
        for (int i = 0; i < kQ8tItemSlots; ++i) {
            mbar_init(&ifull[i], 2);  // item record (producer) and query operand (converter)
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.wfull) + i, 1);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.pnear) + i, 1);  // producer near the item's end
            mbar_init(&iempty[i], 2 * 4 + 2);  // softmax and epilogue warps, S commit, P V thread
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.sfull) + i, 1);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.sfree) + i, 4);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.pfull) + i, 4);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.ofull) + i, 1);
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.ofree) + i, 4);
        }
        for (int i = 0; i < 4; ++i)
            mbar_init(reinterpret_cast<uint64_t *>(smem + L.afull) + i, 4);
        mbar_init(reinterpret_cast<uint64_t *>(smem + L.done), 2 * 4 + 1);
        mbar_init(reinterpret_cast<uint64_t *>(smem + L.fin), 1);
        mbar_init(reinterpret_cast<uint64_t *>(smem + L.fin2), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(reinterpret_cast<uint32_t *>(smem + L.tmem), C::kTmemCols);
        tmem_relinquish();
    }
    // zero the query and P operands: padding columns and other kv heads'
    // entries of P stay zero for the whole kernel
    {
        uint4 *z = reinterpret_cast<uint4 *>(smem + L.qbuf);
        const int n = (kQ8tItemSlots + 2) * kQ8tOp / 16;
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            z[i] = make_uint4(0, 0, 0, 0);
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L.tmem);

    if (warp == 0) {
        q8t_producer<BS, G>(p, &tmk, &tmv, &tsk, &tsv, smem, L);
    } else if (warp == 1) {
        bool ok = true;
        if ((threadIdx.x & 31) == 0) {
            ok = q8t_mma_s<BS, G>(p, smem, L, tmem);
            // every MMA this thread issued has finished before tensor memory goes
            tc_commit(reinterpret_cast<uint64_t *>(smem + L.fin));
            (void)mbar_wait_bounded(reinterpret_cast<uint64_t *>(smem + L.fin), 0);
            if (!ok && p.err)
                atomicOr(p.err, PA_DEVERR_TIMEOUT);
            // the other warps are done with tensor memory
            (void)mbar_wait_bounded(reinterpret_cast<uint64_t *>(smem + L.done), 0);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    } else if (warp == 11) {
        if (!q8t_qconvert<BS, G>(p, smem, L) && (threadIdx.x & 31) == 0 && p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
    } else if (warp == 10) {
        if ((threadIdx.x & 31) == 0) {
            const bool ok = q8t_mma_pv<BS, G>(p, smem, L, tmem);
            tc_commit(reinterpret_cast<uint64_t *>(smem + L.fin2));
            (void)mbar_wait_bounded(reinterpret_cast<uint64_t *>(smem + L.fin2), 0);
            if (!ok && p.err)
                atomicOr(p.err, PA_DEVERR_TIMEOUT);
            tc_fence_before();
            mbar_arrive(reinterpret_cast<uint64_t *>(smem + L.done));
        }
    } else {
        const bool ok = warp < 6 ? q8t_softmax<BS, G>(p, smem, L, tmem) : q8t_epilogue<BS, G>(p, smem, L, tmem);
        if (!ok && (threadIdx.x & 31) == 0 && p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
        tc_fence_before();
        __syncwarp();
        if ((threadIdx.x & 31) == 0)
            mbar_arrive(reinterpret_cast<uint64_t *>(smem + L.done));
    }
    // The CTA has taken its last item: the last CTA to get here returns the
    // launch's counter to zero for the next launch that uses it.
    __syncthreads();
    release_claims(p);
}

}  // namespace pa
