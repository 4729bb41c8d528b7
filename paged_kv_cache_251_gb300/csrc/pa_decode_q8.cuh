// Paged decode attention over an 8-bit KV cache (INT8 or E4M3 codes with one
// fp32 scale per cached row, pa_quant.cuh): the general CUDA-core kernel, any
// query group G in {1, 2, 4, 8}, head_dim 64 or 128, queries in fp32 / fp16 /
// bf16.
//
// Same item structure as the 16-bit general kernel (pa_decode.cuh): items are
// (sequence, kv head, context partition); a producer warp prefetches the
// item's block-table slice and streams, per block, two 1-D bulk copies into a
// stage — the K page and the V page (codes and row scales, pa_quant.cuh) —
// guarded by full/empty mbarriers.
//
// The cached value is code * scale ("KV Cache与长上下文管理", KV-cache
// quantisation; read as per-row scales), so with the codes c_t, c'_t and the
// row scales sk_t, sv_t of token t:
//   x_t   = scale * sk_t * <q, c_t>
//   out   = sum_t e^(x_t - m) sv_t c'_t / sum_t e^(x_t - m)
// Consumers: a row of head_dim codes is split over head_dim / 8 lanes (8 codes
// each, one 8-byte shared load; two rows of 128 codes per warp access cover
// the 32 banks twice, conflict-free); codes are widened exactly to fp32; the
// dot products are reduced with shuffles; each lane group keeps an online
// softmax state for the G heads.
// Every wait is bounded (PA_DEVERR_TIMEOUT); table entries outside the pool
// are never dereferenced (PA_DEVERR_BAD_BLOCK).
#pragma once

#include "pa_decode.cuh"
#include "pa_quant.cuh"

namespace pa {

template <int D, int G> struct Q8Cfg {
    static constexpr int kRow = D;          // bytes of one token's codes
    static constexpr int kEpl = 8;          // codes per lane
    static constexpr int kLpr = D / kEpl;   // lanes per row
    static constexpr int kTpp = 32 / kLpr;  // tokens per warp pass
    static constexpr int kQRowMax = D * 4;  // bytes of one query row (fp32 at most)
    static_assert(kLpr >= 1 && kLpr <= 32 && 32 % kLpr == 0, "a row must map onto whole lanes of a warp");
};

// Stage = [K page][V page].
__host__ __device__ inline uint32_t q8_stage_bytes(int block_size, int D) {
    return 2u * static_cast<uint32_t>(q8_page_bytes(block_size, D));
}

__host__ __device__ inline SmemLayout q8_smem_layout(int S, int block_size, int G, int D) {
    // the 16-bit layout with a stage of q8_stage_bytes and fp32-sized query rows
    return decode_smem_layout(S, q8_stage_bytes(block_size, D) / 2, D * 4, G, D);
}

template <int Fmt, int D, int G>
__device__ inline void q8_producer(const DecodeParams &p, char *smem, const SmemLayout &L) {
    using C = Q8Cfg<D, G>;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    const int bs = p.block_size;
    const uint32_t page = static_cast<uint32_t>(q8_page_bytes(bs, D));
    const uint32_t stage_bytes = q8_stage_bytes(bs, D);
    const uint32_t qrow = static_cast<uint32_t>(D) * (p.q_dtype == PA_F32 ? 4 : 2);
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

    int chunk_base = 0;
    long long chunk_prefix = 0;
    int my_len = 0, my_start = 0, my_np = 0, my_incl = 0, chunk_total = 0;
    bool chunk_ready = false;
    uint32_t t = 0;
    int k = 0;
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
            break;

        const SeqSpan sp = seq_span(len, p.max_len, p.window, bs, p.bpp, start);
        const int blk_lo = sp.b0 + part * p.bpp;
        const int nb = max(0, min(p.bpp, sp.nblk - part * p.bpp));
        const int tok_lo = max(sp.start, blk_lo * bs);
        const int tok_hi = min(sp.end, (blk_lo + nb) * bs);
        const int nst = nb > 0 ? nb : 1;

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
                const uint32_t bytes = (pb >= 0 ? stage_bytes : 0) + (with_q ? G * qrow : 0);
                if (bytes) {
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    if (with_q)
                        bulk_g2s(qbuf + mt.slot * G * C::kQRowMax,
                                 qg + (static_cast<long long>(s) * p.num_heads + kvh * G) * qrow, G * qrow,
                                 &full[stage]);
                    if (pb >= 0) {
                        const long long pix = static_cast<long long>(pb) * p.num_kv_heads + kvh;
                        char *dst = stage_buf + static_cast<size_t>(stage) * stage_bytes;
                        bulk_g2s_hint(dst, kc + pix * page, page, &full[stage], policy);
                        bulk_g2s_hint(dst + page, vc + pix * page, page, &full[stage], policy);
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
            return;
        }
    }
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

template <int Fmt, int D, int G>
__device__ inline void q8_consumer(const DecodeParams &p, char *smem, const SmemLayout &L) {
    using C = Q8Cfg<D, G>;
    constexpr int E = C::kEpl;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gi = lane / C::kLpr;  // token of the pass
    const int li = lane % C::kLpr;  // 8-code chunk of the row
    const int S = p.stages;
    const int bs = p.block_size;
    const uint32_t page = static_cast<uint32_t>(q8_page_bytes(bs, D));
    const uint32_t stage_bytes = q8_stage_bytes(bs, D);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *mfull = reinterpret_cast<uint64_t *>(smem + L.mfull);
    uint64_t *mempty = reinterpret_cast<uint64_t *>(smem + L.mempty);
    const StageMeta *meta = reinterpret_cast<const StageMeta *>(smem + L.meta);
    const ItemInfo *items = reinterpret_cast<const ItemInfo *>(smem + L.items);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.abort);
    const char *qbuf = smem + L.qbuf;
    float *mscr = reinterpret_cast<float *>(smem + L.mscr);
    float *mml = reinterpret_cast<float *>(smem + L.mml);
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
                // the item's G query rows arrived back to back at their own row size
                const int qrow = D * (p.q_dtype == PA_F32 ? 4 : 2);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const char *qr = qbuf + mt.slot * G * C::kQRowMax + g * qrow;
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        qf[g][e] = load_elt(qr, p.q_dtype, li * E + e) * p.scale_log2;
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
            const char *kb = stage_buf + static_cast<size_t>(stage) * stage_bytes;
            const char *vb = kb + page;
            const float *ks = reinterpret_cast<const float *>(kb + bs * C::kRow);  // the pages' scale rows
            const float *vs = reinterpret_cast<const float *>(vb + bs * C::kRow);
            for (int base = warp * C::kTpp; base < mt.hi; base += kConsumerWarps * C::kTpp) {
                const int r = base + gi;
                const bool act = r >= mt.lo && r < mt.hi;
                const int rr = r < bs ? r : bs - 1;  // rows past the block are masked, read in bounds
                float kf[E], vf[E];
                const uint2 kw = ld_shared_v2(kb + rr * C::kRow + li * E);
                Q8<Fmt>::widen4(kw.x, kf);
                Q8<Fmt>::widen4(kw.y, kf + 4);
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
                    sc[g] = x * ks[rr];
                }
                const uint2 vw = ld_shared_v2(vb + rr * C::kRow + li * E);
                Q8<Fmt>::widen4(vw.x, vf);
                Q8<Fmt>::widen4(vw.y, vf + 4);
                const float svr = vs[rr];
                if (act) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float mn = fmaxf(m[g], sc[g]);
                        const float alpha = exp2f(m[g] - mn);
                        const float pw = exp2f(sc[g] - mn);
                        const float pv = pw * svr;
                        l[g] = fmaf(l[g], alpha, pw);
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            acc[g][e] = fmaf(acc[g][e], alpha, pv * vf[e]);
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
                const long long orow = static_cast<long long>(cur.s) * p.num_heads + h;
                if (cur.nparts == 1 && !p.force_partial) {
                    store_out(p.out, p.out_dtype, orow * D + dd, den > 0.f ? num / den : 0.f);
                } else {
                    const long long pr = orow * p.max_parts + cur.part;
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
    if (lane == 0) {
        *abort_flag = 1;
        if (p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
    }
}

template <int Fmt, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads) pa_decode_q8_kernel(const DecodeParams p) {
    // the next kernel on the stream may be launched now (it waits for this
    // grid); this one waits for the kernel before it
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(128) char smem[];
    const SmemLayout L = q8_smem_layout(p.stages, p.block_size, G, D);
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
        q8_producer<Fmt, D, G>(p, smem, L);
    else
        q8_consumer<Fmt, D, G>(p, smem, L);
}

}  // namespace pa
