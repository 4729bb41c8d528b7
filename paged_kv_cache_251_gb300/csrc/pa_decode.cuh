// Paged decode attention: persistent, warp-specialised CUDA-core kernel and
// the log-sum-exp reduce over context partitions.
//
// What it computes ("PagedAttention: From Operating System Virtual Memory to
// Large Language Model Memory Systems", section 2: softmax(Q K^T / sqrt(d)) V;
// "PagedAttention — 把 KV cache 当虚拟内存页来管理", 案例 2: each token's K/V is
// found at (table[t / block_size], t % block_size)): for one query per
// sequence and head, attention over the sequence's attended tokens, with the
// K/V rows read through the block table.
//
// Work unit ("item"): (sequence, kv head, context partition).  A partition is
// up to `bpp` consecutive logical blocks; long contexts are split into
// several partitions whose partial results a second kernel merges by
// log-sum-exp (the mjmagnets article, section 2.2: a long sequence becomes
// several attention units).
//
// CTA = 1 producer warp + 4 consumer warps; the grid is persistent (a few
// CTAs per SM, each walking items blockIdx.x, blockIdx.x + gridDim.x, ...).
//  - producer: for its next item, loads the item's slice of the block table
//    into shared memory (one coalesced read, entries range-checked), then for
//    each block issues two 1-D bulk copies (TMA) of the contiguous
//    (block, kv head) K and V tiles into a ring of `stages` buffers guarded
//    by full/empty mbarriers; the first stage of an item also brings the
//    item's G query rows.  The producer runs ahead across item boundaries.
//  - consumers: each stage's tokens are split over the 4 warps; inside a warp
//    a group of row_bytes / 16 lanes owns one token (16-byte shared loads,
//    one lane per 16 bytes of the row).  Scores are fp32 dot products reduced
//    with warp shuffles; each group keeps an online-softmax state (running
//    max m, denominator l, fp32 accumulator) for the G heads of the group.
//    At an item's last stage the groups and warps merge their states and the
//    item writes either the final output row (single-partition sequence) or
//    its partial (m, l, unnormalised accumulator) to the workspace.
// Every wait is bounded (about 2 s, then PA_DEVERR_TIMEOUT); table entries
// outside the pool are never dereferenced (PA_DEVERR_BAD_BLOCK, tokens left
// out of the softmax).
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxBpp = 256;  // blocks per partition (table-slice capacity)

struct DecodeParams {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *part_acc;  // [N][H][max_parts][D]
    float *part_ml;   // [N][H][max_parts][2]: running max (log2 units), denominator
    uint32_t *err;
    int num_seqs, num_heads, num_kv_heads, block_size, window;
    int max_blocks_per_seq, num_blocks, bpp, max_parts, out_dtype, stages;
    int max_len;       // max_blocks_per_seq * block_size
    float scale_log2;  // scale * log2(e): scores are kept in base-2 units
    const int32_t *start_tok;  // per-sequence first attended token (nullable)
    int force_partial;         // 1: always write partials, even for one partition
    // 8-bit caches only: the element type of q (the caches hold pages of
    // codes and row scales)
    int q_dtype;
    // Dynamic item scheduling (kernels that support it): {next item, CTAs
    // done}, zero before the launch and returned to zero by its last CTA;
    // nullptr: items go round-robin over the CTAs.
    unsigned int *work = nullptr;
    // 1: the caches are contiguous, [num_seqs][num_kv_heads][max_len][D]
    // (no block table: block b of sequence s and kv head h is tile
    // (s * num_kv_heads + h) * max_blocks_per_seq + b); the MHA and
    // tensor-core grouped-head kernels only
    int contiguous = 0;
};

// Tile index (into the [tiles][block_size][D] view of a cache) of table entry
// or logical block `pb` of sequence s and kv head h.
__device__ inline int kv_tile(const DecodeParams &p, int s, int h, int pb) {
    return p.contiguous ? (s * p.num_kv_heads + h) * p.max_blocks_per_seq + pb : pb * p.num_kv_heads + h;
}

// Items of a persistent decode kernel, for its producer warp: from the
// launch's counter (DecodeParams::work), or round-robin without one.  A CTA's
// first item is its own (no round trip before the first copy); the counter
// numbers the later ones from gridDim.x up.  The kernel claims the item after
// the current one with claim_next when the current one has a few copies left
// to issue (next claims it on demand otherwise): a claim taken earlier would
// sit unstarted, and at the end of a launch the CTAs holding one would finish
// an item's time after the rest.  Claimed indices only grow, so the producer's
// forward scan over the contexts still applies; every claimed index below the
// item count is processed.
struct ItemClaim {
    long long w = 0;         // the current item
    unsigned int ahead = 0;  // the next one (lane 0)
    bool claimed = false;    // `ahead` holds a claim (warp-uniform)
    __device__ void start() {
        w = blockIdx.x;
        claimed = false;
    }
    // claim the item after the current one now (once)
    __device__ void claim_next(const DecodeParams &p) {
        const int lane = threadIdx.x & 31;
        if (p.work && !claimed) {
            if (lane == 0)
                ahead = gridDim.x + atomicAdd(p.work, 1u);
            claimed = true;
        }
    }
    __device__ void next(const DecodeParams &p) {
        if (p.work) {
            claim_next(p);
            w = __shfl_sync(0xffffffffu, ahead, 0);
            claimed = false;
        } else {
            w += gridDim.x;
        }
    }
    // the claims are complete before the CTA reports itself done
    __device__ void finish(const DecodeParams &p) const {
        if (p.work)
            __threadfence();
    }
};

// The item order of the persistent kernels: (sequence, context partition)
// pairs in sequence order, each taken with every kv head (or kv-head group).
// Item f is found by a forward scan over context_lens, 32 sequences at a
// time; a CTA's item indices only grow, so the scan never moves backwards.
// (An order with every full partition first and the partial ones last was
// measured: it shortens the end of a launch but puts the items with the
// largest fixed cost per byte back to back, and was slower on the GQA batch.)
struct ItemScan {
    int chunk_base = 0;
    long long chunk_prefix = 0;
    int my_len = 0, my_start = 0, my_np = 0, my_incl = 0, chunk_total = 0;
    bool chunk_ready = false;

    // The sequence of item f (-1 past the last item), with its partition, its
    // context length and its first attended token.  Warp-collective.
    __device__ int find(const DecodeParams &p, int block_size, long long f, int &part, int &len, int &start) {
        const int lane = threadIdx.x & 31;
        for (;;) {
            if (!chunk_ready) {
                if (chunk_base >= p.num_seqs)
                    return -1;
                const int sq = chunk_base + lane;
                my_len = sq < p.num_seqs ? ld_nc_i32(p.context_lens + sq) : 0;
                if (sq < p.num_seqs && my_len > p.max_len && p.err)
                    atomicOr(p.err, PA_DEVERR_BAD_LEN);
                my_start = (sq < p.num_seqs && p.start_tok) ? ld_nc_i32(p.start_tok + sq) : 0;
                my_np = sq < p.num_seqs ? seq_span(my_len, p.max_len, p.window, block_size, p.bpp, my_start).nparts : 0;
                my_incl = my_np;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, my_incl, o);
                    if (lane >= o)
                        my_incl += v;
                }
                chunk_total = __shfl_sync(0xffffffffu, my_incl, 31);
                chunk_ready = true;
            }
            if (f < chunk_prefix + chunk_total) {
                const unsigned hit = __ballot_sync(0xffffffffu, chunk_prefix + my_incl > f);
                const int j = __ffs(hit) - 1;
                const int incl_j = __shfl_sync(0xffffffffu, my_incl, j);
                const int np_j = __shfl_sync(0xffffffffu, my_np, j);
                len = __shfl_sync(0xffffffffu, my_len, j);
                start = __shfl_sync(0xffffffffu, my_start, j);
                part = static_cast<int>(f - (chunk_prefix + incl_j - np_j));
                return chunk_base + j;
            }
            chunk_prefix += chunk_total;
            chunk_base += 32;
            chunk_ready = false;
        }
    }
};

// A producer's next item, found and its block-table slice loaded into
// registers one item ahead: the scan's and the table's memory latency then
// overlaps the current item's copies instead of stalling the stage ring.
struct NextItem {
    int s, part, len, start, head;  // head: kv head, or kv-head group, of the item
    SeqSpan sp;
    int blk_lo, nb;
    int tb[kMaxBpp / 32];  // table entry lane + 32 i of the slice (checked when stored)
};

// Item w of the order (w / groups, head w % groups); warp-collective.
__device__ inline void prepare_item(const DecodeParams &p, int block_size, ItemScan &scan, long long w,
                                    long long groups, NextItem &n) {
    const int lane = threadIdx.x & 31;
    n.head = static_cast<int>(w % groups);
    n.part = n.len = n.start = 0;
    n.s = scan.find(p, block_size, w / groups, n.part, n.len, n.start);
    n.blk_lo = n.nb = 0;
    if (n.s < 0)
        return;
    n.sp = seq_span(n.len, p.max_len, p.window, block_size, p.bpp, n.start);
    n.blk_lo = n.sp.b0 + n.part * p.bpp;
    n.nb = max(0, min(p.bpp, n.sp.nblk - n.part * p.bpp));
    const int32_t *row = p.block_tables + static_cast<long long>(n.s) * p.max_blocks_per_seq + n.blk_lo;
#pragma unroll
    for (int i = 0; i < kMaxBpp / 32; ++i) {
        const int j = lane + 32 * i;
        n.tb[i] = j < n.nb ? (p.contiguous ? n.blk_lo + j : ld_nc_i32(row + j)) : -1;
    }
}

// The item's table slice into shared memory; entries outside the pool become
// -1 and are flagged (PA_DEVERR_BAD_BLOCK).
__device__ inline void store_table(const DecodeParams &p, const NextItem &n, int32_t *tbl) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < kMaxBpp / 32; ++i) {
        const int j = lane + 32 * i;
        if (j < n.nb) {
            int pb = n.tb[i];
            if (pb < 0 || pb >= p.num_blocks) {
                pb = -1;
                if (p.err)
                    atomicOr(p.err, PA_DEVERR_BAD_BLOCK);
            }
            tbl[j] = pb;
        }
    }
}

// End of a launch with claimed items, once every thread of the CTA is past its
// last claim (the caller synchronises the CTA first): the last CTA returns the
// counter pair to zero for the next launch that uses it.
__device__ inline void release_claims(const DecodeParams &p) {
    if (threadIdx.x == 0 && p.work) {
        __threadfence();
        if (atomicAdd(p.work + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.work, 0u);
            atomicExch(p.work + 1, 0u);
        }
    }
}

struct StageMeta {
    int slot;   // item slot (item counter mod stages)
    int lo;     // first attended row of the block
    int hi;     // one past the last attended row
    int flags;  // kValid | kFirst | kLast | kEnd | kHasQ
};
constexpr int kValid = 1, kFirst = 2, kLast = 4, kEnd = 8, kHasQ = 16;

struct ItemInfo {
    int s, kvh, part, nparts;
};

struct SmemLayout {
    uint32_t full, empty, mfull, mempty, meta, items, abort, table, qbuf, mscr, mml, stages, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SmemLayout decode_smem_layout(int S, int tile_bytes, int row_bytes, int G,
                                                         int D) {
    SmemLayout L;
    uint32_t off = 0;
    L.full = off;
    off += 8 * S;
    L.empty = off;
    off += 8 * S;
    L.mfull = off;
    off += 16;
    L.mempty = off;
    off += 16;
    L.meta = align_up(off, 16);
    off = L.meta + 16 * S;
    L.items = off;
    off += 16 * S;
    L.abort = off;
    off += 16;
    L.table = off;
    off += 4 * kMaxBpp;
    L.qbuf = align_up(off, 128);
    off = L.qbuf + S * G * row_bytes;
    L.mscr = align_up(off, 16);
    off = L.mscr + 2 * kConsumerWarps * G * D * 4;
    L.mml = off;
    off += 2 * kConsumerWarps * G * 2 * 4;
    L.stages = align_up(off, 128);
    off = L.stages + S * 2 * tile_bytes;
    L.total = off;
    return L;
}

template <typename T, int D, int G> struct DecodeCfg {
    static constexpr int kElt = sizeof(T);
    static constexpr int kRow = D * kElt;    // bytes of one token's K (or V) row
    static constexpr int kLpr = kRow / 16;   // lanes per row
    static constexpr int kEpl = 16 / kElt;   // elements per lane
    static constexpr int kTpp = 32 / kLpr;   // tokens per warp pass
    static_assert(kLpr >= 1 && kLpr <= 32 && 32 % kLpr == 0, "a row must map onto whole lanes of a warp");
};

// Merge an online-softmax state (m, l, acc) with another (mo, lo, acco).
template <int E>
__device__ inline void merge_state(float &m, float &l, float *acc, float mo, float lo, const float *acco) {
    const float M = fmaxf(m, mo);
    if (M == -INFINITY)
        return;
    const float a = exp2f(m - M), b = exp2f(mo - M);
    l = l * a + lo * b;
#pragma unroll
    for (int e = 0; e < E; ++e)
        acc[e] = acc[e] * a + acco[e] * b;
    m = M;
}

template <typename T, int D, int G>
__device__ inline void decode_producer(const DecodeParams &p, char *smem, const SmemLayout &L) {
    using C = DecodeCfg<T, D, G>;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    const int bs = p.block_size;
    const uint32_t tile = static_cast<uint32_t>(bs) * C::kRow;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + L.meta);
    ItemInfo *items = reinterpret_cast<ItemInfo *>(smem + L.items);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.abort);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + L.table);
    char *qbuf = smem + L.qbuf;
    char *stage_buf = smem + L.stages;
    const char *kc = static_cast<const char *>(p.k_cache);
    const char *vc = static_cast<const char *>(p.v_cache);
    const char *qg = static_cast<const char *>(p.q);
    const uint64_t policy = policy_evict_first();

    // Sequences are scanned 32 at a time: lane j holds sequence chunk_base + j.
    int chunk_base = 0;
    long long chunk_prefix = 0;  // partitions of all sequences before chunk_base
    int my_len = 0, my_start = 0, my_np = 0, my_incl = 0, chunk_total = 0;
    bool chunk_ready = false;

    uint32_t t = 0;  // stages issued
    int k = 0;       // items issued
    bool ok = true;
    const long long hkv = p.num_kv_heads;

    for (long long w = blockIdx.x; ok; w += gridDim.x) {
        const long long f = w / hkv;
        const int kvh = static_cast<int>(w % hkv);
        int s = -1, part = 0, len = 0, start = 0, nparts = 1;
        for (;;) {
            if (!chunk_ready) {
                if (chunk_base >= p.num_seqs)
                    break;
                const int sq = chunk_base + lane;
                my_len = sq < p.num_seqs ? ld_nc_i32(p.context_lens + sq) : 0;
                if (sq < p.num_seqs && my_len > p.max_len && p.err)
                    atomicOr(p.err, PA_DEVERR_BAD_LEN);
                my_start = (sq < p.num_seqs && p.start_tok) ? ld_nc_i32(p.start_tok + sq) : 0;
                my_np = sq < p.num_seqs ? seq_span(my_len, p.max_len, p.window, bs, p.bpp, my_start).nparts : 0;
                my_incl = my_np;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, my_incl, o);
                    if (lane >= o)
                        my_incl += v;
                }
                chunk_total = __shfl_sync(0xffffffffu, my_incl, 31);
                chunk_ready = true;
            }
            if (f < chunk_prefix + chunk_total) {
                const unsigned hit = __ballot_sync(0xffffffffu, chunk_prefix + my_incl > f);
                const int j = __ffs(hit) - 1;
                s = chunk_base + j;
                const int incl_j = __shfl_sync(0xffffffffu, my_incl, j);
                nparts = __shfl_sync(0xffffffffu, my_np, j);
                len = __shfl_sync(0xffffffffu, my_len, j);
                start = __shfl_sync(0xffffffffu, my_start, j);
                part = static_cast<int>(f - (chunk_prefix + incl_j - nparts));
                break;
            }
            chunk_prefix += chunk_total;
            chunk_base += 32;
            chunk_ready = false;
        }
        if (s < 0)
            break;  // no more items for this CTA

        const SeqSpan sp = seq_span(len, p.max_len, p.window, bs, p.bpp, start);
        const int blk_lo = sp.b0 + part * p.bpp;
        const int nb = max(0, min(p.bpp, sp.nblk - part * p.bpp));
        const int tok_lo = max(sp.start, blk_lo * bs);
        const int tok_hi = min(sp.end, (blk_lo + nb) * bs);
        const int nst = nb > 0 ? nb : 1;

        // Block-table slice of this item -> shared memory (entries checked).
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

        for (int j = 0; j < nst; ++j, ++t) {
            const int stage = static_cast<int>(t % S);
            const uint32_t par = ((t / S) & 1u) ^ 1u;
            if (*abort_flag || !mbar_wait_bounded(&empty[stage], par)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const int pb = nb > 0 ? tbl[j] : -1;
                int lo = 0, hi = 0;
                if (nb > 0) {
                    const int blk = blk_lo + j;
                    lo = max(tok_lo - blk * bs, 0);
                    hi = min(tok_hi - blk * bs, bs);
                }
                StageMeta mt;
                mt.slot = k % S;
                mt.lo = lo;
                mt.hi = hi;
                const bool with_q = (j == 0 && nb > 0);
                mt.flags = (pb >= 0 ? kValid : 0) | (j == 0 ? kFirst : 0) | (j == nst - 1 ? kLast : 0) |
                           (with_q ? kHasQ : 0);
                meta[stage] = mt;
                if (j == 0) {
                    ItemInfo it;
                    it.s = s;
                    it.kvh = kvh;
                    it.part = part;
                    it.nparts = sp.nparts;
                    items[mt.slot] = it;
                }
                const uint32_t bytes = (pb >= 0 ? 2 * tile : 0) + (with_q ? G * C::kRow : 0);
                if (bytes) {
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    if (with_q)
                        bulk_g2s(qbuf + mt.slot * G * C::kRow,
                                 qg + (static_cast<long long>(s) * p.num_heads + kvh * G) * C::kRow,
                                 G * C::kRow, &full[stage]);
                    if (pb >= 0) {
                        const long long off = (static_cast<long long>(pb) * p.num_kv_heads + kvh) * tile;
                        char *dst = stage_buf + static_cast<size_t>(stage) * 2 * tile;
                        bulk_g2s_hint(dst, kc + off, tile, &full[stage], policy);
                        bulk_g2s_hint(dst + tile, vc + off, tile, &full[stage], policy);
                    }
                } else {
                    mbar_arrive(&full[stage]);
                }
            }
            __syncwarp();
        }
        ++k;
    }

    if (ok) {
        // End marker: one more stage that carries no data.
        const int stage = static_cast<int>(t % S);
        const uint32_t par = ((t / S) & 1u) ^ 1u;
        if (!*abort_flag && mbar_wait_bounded(&empty[stage], par)) {
            if (lane == 0) {
                StageMeta mt;
                mt.slot = 0;
                mt.lo = mt.hi = 0;
                mt.flags = kEnd;
                meta[stage] = mt;
                mbar_arrive(&full[stage]);
            }
            __syncwarp();
            ++t;
            return;
        }
    }
    // Give up: flag it, then wait (bounded) for our copies still in flight so
    // no bulk copy lands in shared memory after the CTA has gone.
    if (lane == 0) {
        *abort_flag = 1;
        if (p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
        const uint32_t first = t > static_cast<uint32_t>(S) ? t - S : 0;
        for (uint32_t u = first; u < t; ++u)
            (void)mbar_wait_bounded(&full[u % S], (u / S) & 1u);
    }
    __syncwarp();
}

template <typename T, int D, int G>
__device__ inline void decode_consumer(const DecodeParams &p, char *smem, const SmemLayout &L) {
    using C = DecodeCfg<T, D, G>;
    constexpr int E = C::kEpl;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gi = lane / C::kLpr;  // token group inside the warp
    const int li = lane % C::kLpr;  // 16-byte chunk of the row
    const int S = p.stages;
    const uint32_t tile = static_cast<uint32_t>(p.block_size) * C::kRow;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *mfull = reinterpret_cast<uint64_t *>(smem + L.mfull);
    uint64_t *mempty = reinterpret_cast<uint64_t *>(smem + L.mempty);
    const StageMeta *meta = reinterpret_cast<const StageMeta *>(smem + L.meta);
    const ItemInfo *items = reinterpret_cast<const ItemInfo *>(smem + L.items);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.abort);
    const char *qbuf = smem + L.qbuf;
    float *mscr = reinterpret_cast<float *>(smem + L.mscr);  // [2][warps][G][D]
    float *mml = reinterpret_cast<float *>(smem + L.mml);    // [2][warps][G][2]
    const char *stage_buf = smem + L.stages;

    float qf[G][E];
    float m[G], l[G], acc[G][E];
    ItemInfo cur = {0, 0, 0, 1};

    uint32_t t = 0;
    int k = 0;
    for (;;) {
        const int stage = static_cast<int>(t % S);
        if (!mbar_wait_bounded(&full[stage], (t / S) & 1u))
            break;
        const StageMeta mt = meta[stage];
        if (mt.flags & kEnd)
            return;
        if (mt.flags & kFirst) {
            cur = items[mt.slot];
            if (mt.flags & kHasQ) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const uint4 r = ld_shared_v4(qbuf + (mt.slot * G + g) * C::kRow + li * 16);
                    Elt<T>::unpack(r, qf[g]);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        qf[g][e] *= p.scale_log2;
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                m[g] = -INFINITY;
                l[g] = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e)
                    acc[g][e] = 0.f;
            }
        }
        if (mt.flags & kValid) {
            const char *kb = stage_buf + static_cast<size_t>(stage) * 2 * tile;
            const char *vb = kb + tile;
            for (int base = warp * C::kTpp; base < mt.hi; base += kConsumerWarps * C::kTpp) {
                const int r = base + gi;
                const bool act = r >= mt.lo && r < mt.hi;
                float kf[E], vf[E];
                Elt<T>::unpack(ld_shared_v4(kb + r * C::kRow + li * 16), kf);
                float sc[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float x = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        x = fmaf(qf[g][e], kf[e], x);
#pragma unroll
                    for (int o = C::kLpr / 2; o > 0; o >>= 1)
                        x += __shfl_xor_sync(0xffffffffu, x, o);
                    sc[g] = x;
                }
                Elt<T>::unpack(ld_shared_v4(vb + r * C::kRow + li * 16), vf);
                if (act) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float mn = fmaxf(m[g], sc[g]);
                        const float alpha = exp2f(m[g] - mn);
                        const float pw = exp2f(sc[g] - mn);
                        l[g] = fmaf(l[g], alpha, pw);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            acc[g][e] = fmaf(acc[g][e], alpha, pw * vf[e]);
                        m[g] = mn;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);
        ++t;

        if (mt.flags & kLast) {
            // 1) merge the token groups of this warp
#pragma unroll
            for (int o = C::kLpr; o < 32; o <<= 1) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float ao[E];
                    const float mo = __shfl_xor_sync(0xffffffffu, m[g], o);
                    const float lo = __shfl_xor_sync(0xffffffffu, l[g], o);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        ao[e] = __shfl_xor_sync(0xffffffffu, acc[g][e], o);
                    merge_state<E>(m[g], l[g], acc[g], mo, lo, ao);
                }
            }
            // 2) publish this warp's state, double-buffered by item parity
            const int b = k & 1;
            const uint32_t use = static_cast<uint32_t>(k >> 1) & 1u;
            if (!mbar_wait_bounded(&mempty[b], use ^ 1u))
                break;
            if (gi == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        mscr[((b * kConsumerWarps + warp) * G + g) * D + li * E + e] = acc[g][e];
                    if (li == 0) {
                        mml[((b * kConsumerWarps + warp) * G + g) * 2 + 0] = m[g];
                        mml[((b * kConsumerWarps + warp) * G + g) * 2 + 1] = l[g];
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&mfull[b]);
            if (!mbar_wait_bounded(&mfull[b], use))
                break;
            // 3) combine the warps; each consumer thread finishes some (head, dim)
            const int ctid = warp * 32 + lane;
            for (int idx = ctid; idx < G * D; idx += kConsumerWarps * 32) {
                const int g = idx / D, dd = idx % D;
                float M = -INFINITY;
#pragma unroll
                for (int w2 = 0; w2 < kConsumerWarps; ++w2)
                    M = fmaxf(M, mml[((b * kConsumerWarps + w2) * G + g) * 2]);
                float num = 0.f, den = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
                        const float mw = mml[((b * kConsumerWarps + w2) * G + g) * 2];
                        const float sc = exp2f(mw - M);
                        num = fmaf(mscr[((b * kConsumerWarps + w2) * G + g) * D + dd], sc, num);
                        den = fmaf(mml[((b * kConsumerWarps + w2) * G + g) * 2 + 1], sc, den);
                    }
                }
                const int h = cur.kvh * G + g;
                const long long row = static_cast<long long>(cur.s) * p.num_heads + h;
                if (cur.nparts == 1 && !p.force_partial) {
                    store_out(p.out, p.out_dtype, row * D + dd, den > 0.f ? num / den : 0.f);
                } else {
                    const long long pr = row * p.max_parts + cur.part;
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
            ++k;
        }
    }
    // a wait gave up
    if (lane == 0) {
        *abort_flag = 1;
        if (p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
    }
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads) pa_decode_kernel(const DecodeParams p) {
    // the next kernel on the stream may be launched now (it waits for this
    // grid); this one waits for the kernel before it
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(128) char smem[];
    using C = DecodeCfg<T, D, G>;
    const SmemLayout L = decode_smem_layout(p.stages, p.block_size * C::kRow, C::kRow, G, D);
    if (threadIdx.x == 0) {
        uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
        uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        uint64_t *mfull = reinterpret_cast<uint64_t *>(smem + L.mfull);
        uint64_t *mempty = reinterpret_cast<uint64_t *>(smem + L.mempty);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&mfull[i], kConsumerWarps);
            mbar_init(&mempty[i], kConsumerWarps);
        }
        *reinterpret_cast<int *>(smem + L.abort) = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if ((threadIdx.x >> 5) == kConsumerWarps)
        decode_producer<T, D, G>(p, smem, L);
    else
        decode_consumer<T, D, G>(p, smem, L);
}

// Merge the partitions of every multi-partition (sequence, head):
//   M = max_p m_p,  out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p
// Two layouts: pa_reduce_kernel, one warp per (sequence, head) row and
// kReduceRows rows per CTA with no CTA-wide step (the lanes take the (m, l)
// pairs for the row max and the denominator, then each lane sums its head_dim
// slice over the partitions, the loads of several partitions in flight), for
// many rows of few partitions; pa_reduce_wide_kernel, one CTA per row (the
// warps take partitions round-robin, each merges its own with a running max,
// and the warps' results are merged through shared memory), for few rows of
// many partitions.  Single-partition rows were written by the decode kernel
// and are left alone.
constexpr int kReduceThreads = 128;
constexpr int kReduceWideThreads = 256;
constexpr int kReduceRows = kReduceThreads / 32;

template <int D>
__global__ void __launch_bounds__(kReduceThreads) pa_reduce_kernel(const DecodeParams p) {
    // (the host takes this layout only for max_parts <= 32: lane q holds partition q)
    pdl_launch_dependents();
    pdl_wait();
    constexpr int kPer = D / 32;  // head_dim slice per lane (4 or 2)
    constexpr int kBatch = 8;     // partitions whose slices are loaded before any is used
    const int lane = threadIdx.x & 31;
    const long long rowi = static_cast<long long>(blockIdx.x) * kReduceRows + (threadIdx.x >> 5);
    if (rowi >= static_cast<long long>(p.num_seqs) * p.num_heads)
        return;
    const int s = static_cast<int>(rowi / p.num_heads);
    const long long base = rowi * p.max_parts;
    // the context length and every partition's (m, l) in one round trip
    const int len = ld_nc_i32(p.context_lens + s);
    const int start = p.start_tok ? ld_nc_i32(p.start_tok + s) : 0;
    float2 mine = make_float2(-INFINITY, 0.f);
    if (lane < p.max_parts)
        mine = reinterpret_cast<const float2 *>(p.part_ml + base * 2)[lane];
    const SeqSpan sp = seq_span(len, p.max_len, p.window, p.block_size, p.bpp, start);
    const int np = sp.nparts;
    if (np <= 1)
        return;
    if (lane >= np)
        mine = make_float2(-INFINITY, 0.f);  // stale entries of unused partitions
    float M = mine.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float sc = (M == -INFINITY || mine.x == -INFINITY) ? 0.f : exp2f(mine.x - M);
    float den = mine.y * sc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        den += __shfl_xor_sync(0xffffffffu, den, o);

    float num[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        num[i] = 0.f;
    const float *a = p.part_acc + base * D + lane * kPer;
    for (int q0 = 0; q0 < np; q0 += kBatch) {
        float v[kBatch][kPer];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (q0 + j < np) {
                if constexpr (kPer == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(a + static_cast<long long>(q0 + j) * D);
                    v[j][0] = x.x, v[j][1] = x.y, v[j][2] = x.z, v[j][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(a + static_cast<long long>(q0 + j) * D);
                    v[j][0] = x.x, v[j][1] = x.y;
                }
            } else {
#pragma unroll
                for (int i = 0; i < kPer; ++i)
                    v[j][i] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const float scj = __shfl_sync(0xffffffffu, sc, (q0 + j) & 31);
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                num[i] = fmaf(v[j][i], scj, num[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        store_out(p.out, p.out_dtype, rowi * D + lane * kPer + i, den > 0.f ? num[i] / den : 0.f);
}

template <int D>
__global__ void __launch_bounds__(kReduceWideThreads) pa_reduce_wide_kernel(const DecodeParams p) {
    pdl_launch_dependents();
    pdl_wait();
    constexpr int kWarps = kReduceWideThreads / 32;
    constexpr int kPer = D / 32;  // head_dim slice per lane (4 or 2)
    constexpr int kBatch = 8;     // partitions of one warp whose slices are loaded before any is used
    constexpr int kStep = kWarps * kBatch;
    __shared__ float wmax[kWarps], wden[kWarps];
    __shared__ float accs[kWarps][D];
    const long long rowi = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = static_cast<int>(rowi / p.num_heads);
    const long long base = rowi * p.max_parts;
    const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml + base * 2);
    const float *acc = p.part_acc + base * D + lane * kPer;

    // warp w takes partitions w, w + kWarps, ...; a batch is kBatch of them
    float2 m[kBatch];
    float v[kBatch][kPer];
    auto load = [&](int q0, int lim) {
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int q = q0 + warp + kWarps * j;
            m[j] = make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                v[j][i] = 0.f;
            if (q < lim) {
                m[j] = ml[q];
                if constexpr (kPer == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(acc + static_cast<long long>(q) * D);
                    v[j][0] = x.x, v[j][1] = x.y, v[j][2] = x.z, v[j][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(acc + static_cast<long long>(q) * D);
                    v[j][0] = x.x, v[j][1] = x.y;
                }
            }
        }
    };
    // the context length and the first batch in one round trip: the batch is
    // bounded by the workspace's partitions per row, entries past the row's
    // own partitions are dropped below
    const int len = ld_nc_i32(p.context_lens + s);
    const int start = p.start_tok ? ld_nc_i32(p.start_tok + s) : 0;
    load(0, p.max_parts);
    const SeqSpan sp = seq_span(len, p.max_len, p.window, p.block_size, p.bpp, start);
    const int np = sp.nparts;
    if (np <= 1)
        return;

    // this warp's running max, denominator and numerator slice
    float mw = -INFINITY, dw = 0.f, nw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        nw[i] = 0.f;
    for (int q0 = 0;; q0 += kStep) {
        float bm = -INFINITY;
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (q0 + warp + kWarps * j < np)
                bm = fmaxf(bm, m[j].x);
        const float mn = fmaxf(mw, bm);
        if (mn != -INFINITY) {
            const float a = mw == -INFINITY ? 0.f : exp2f(mw - mn);
            dw *= a;
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                nw[i] *= a;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (q0 + warp + kWarps * j < np && m[j].x != -INFINITY) {
                    const float sc = exp2f(m[j].x - mn);
                    dw = fmaf(m[j].y, sc, dw);
#pragma unroll
                    for (int i = 0; i < kPer; ++i)
                        nw[i] = fmaf(v[j][i], sc, nw[i]);
                }
            }
            mw = mn;
        }
        if (q0 + kStep >= np)
            break;
        load(q0 + kStep, np);
    }
    if (lane == 0) {
        wmax[warp] = mw;
        wden[warp] = dw;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        accs[warp][lane * kPer + i] = nw[i];
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
        M = fmaxf(M, wmax[w]);
    for (int d = tid; d < D; d += kReduceWideThreads) {
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float sc = wmax[w] == -INFINITY ? 0.f : exp2f(wmax[w] - M);
                num = fmaf(accs[w][d], sc, num);
                den = fmaf(wden[w], sc, den);
            }
        }
        store_out(p.out, p.out_dtype, rowi * D + d, den > 0.f ? num / den : 0.f);
    }
}

}  // namespace pa
