// Paged decode attention over an 8-bit KV cache, head_dim 128, query groups
// G in {1, 2, 4}: the persistent, warp-specialised kernel fed by TMA tensor
// copies (the 16-bit MHA kernel's data path, pa_decode_mha.cuh), with
// arithmetic chosen for 1-byte elements.
//
// What it computes is pa_decode's attention with every cached element read as
// code * scale of its row (pa_quant.cuh): for token t of a sequence with codes
// c_t, c'_t and row scales sk_t, sv_t,
//   x_t = scale * sk_t * <q, c_t>,  out = sum_t e^(x_t - m) sv_t c'_t / sum_t e^(x_t - m).
//
// Data path: per (block, kv head) one 1-D bulk copy of the K page and one of
// the V page (block_size code rows of 128 bytes, then a row of fp32 scales:
// pa_quant.cuh) into a ring of stages owned round-robin by the 4 consumer
// warps (stage t belongs to warp t % 4; the ring length is a multiple of 4).
// Items (sequence, kv head, partition) flow through a 4-slot ring; each
// item's G query rows ride on its item barrier.
//
// Consumers: a warp is G head groups of W = 32 / G lanes; each lane serves one
// query head through the whole item (its own running max, denominator and
// accumulator), so every reduction stays inside a head group.  Per block of
// block_size tokens:
//  - QK: a head group's lanes are (token, part) pairs, kTpr tokens per round
//    and kP = W / kTpr lanes per token (a 128-code row split kP ways).
//      INT8: the query row is quantised once per item to int16 (scale
//      max|q| / 32767) and dp2a multiplies 16-bit query pairs by code bytes
//      exactly into int32 sums.
//      E4M3: codes are widened pairwise to fp16 (cvt e4m3x2 -> f16x2, exact)
//      and multiplied by the query in fp16 (scaled by a power of two, so the
//      conversion of fp16 / bf16 queries is exact), fp32 accumulation.
//  - softmax at block granularity: one running-max update per block.
//  - PV: each lane owns 4G consecutive output dimensions of its head.
//      INT8: the block's weights p_t * sv_t are quantised to int16 (scale: the
//      block's largest weight / 32767), pairs of tokens are byte-interleaved
//      with one permute per 4 dimensions, and dp2a accumulates both tokens of
//      a dimension in one instruction; the int32 sums join the fp32
//      accumulator once per block.
//      E4M3: codes widened to fp32, fp32 FMA with the fp32 weight.
//  Pages land unswizzled: in QK the lanes of one token row read its chunks in
//  an order rotated by the token index (their query pairs are stored rotated
//  the same way), so each shared load spreads over all 32 banks; in PV all
//  lanes read one row.  Shared-memory offsets are per-lane constants, stage
//  indices advance without division.
// Every wait is bounded (PA_DEVERR_TIMEOUT); table entries outside the pool
// are never dereferenced (PA_DEVERR_BAD_BLOCK).
#pragma once

#include "pa_decode.cuh"
#include "pa_quant.cuh"

namespace pa {

constexpr int kQ8fWarps = 4;
constexpr int kQ8fThreads = (kQ8fWarps + 1) * 32;
constexpr int kQ8fItemSlots = 4;
constexpr int kQ8fD = 128;

struct Q8fItem {
    int s, kvh, part, nparts;
    int nb;       // blocks of the item (0: empty sequence)
    int tok_lo;   // attended tokens of the item: [tok_lo, tok_hi)
    int tok_hi;
    int blk_lo;   // first logical block
    int t_first;  // pipeline stage of the first block
    int end;      // 1: no more items
    int pad[2];
};

template <int G, int BS> struct Q8fCfg {
    static constexpr int D = kQ8fD;
    static constexpr int kW = 32 / G;                                   // lanes per head group
    // lanes per token in QK: a token's 128 codes over 2 lanes (G <= 2 with a
    // 16-token round, G = 4), 4 lanes at block size 8 (G = 1), 1 lane for
    // G = 2 at 16 tokens a round
    static constexpr int kP = G == 4 ? 2 : (G == 2 ? (BS < 16 ? 2 : 1) : (BS < 16 ? 4 : 2));
    static constexpr int kTpr = kW / kP;                                // tokens per QK round
    static constexpr int kRounds = BS / kTpr;
    static constexpr int kCpl = 8 / kP;                                 // 16-byte code chunks per QK lane
    static constexpr int kQp = 64 / kP;                                 // packed query pairs per lane
    static constexpr int kDG = 4 * G;                                   // PV dims per lane
    static constexpr int kPage = q8_page_bytes(BS, D);                  // bytes of one page
    static constexpr int kQRow = D * 4;                                 // query row slot (fp32 at most)
    static_assert(kTpr % 2 == 0 && kP >= 1 && kCpl >= 1 && BS % kTpr == 0, "lane mapping");
};

struct Q8fLayout {
    uint32_t full, empty, ifull, iempty, mfull, mempty, valid, items, table, qbuf, mscr, mml, stages, total;
};

__host__ __device__ inline Q8fLayout q8f_smem_layout(int S, int BS, int G) {
    Q8fLayout L;
    uint32_t off = 0;
    L.full = off;
    off += 8 * S;
    L.empty = off;
    off += 8 * S;
    L.ifull = off;
    off += 8 * kQ8fItemSlots;
    L.iempty = off;
    off += 8 * kQ8fItemSlots;
    L.mfull = off;
    off += 16;
    L.mempty = off;
    off += 16;
    L.valid = off;
    off += 4 * S;
    L.items = align_up(off, 16);
    off = L.items + sizeof(Q8fItem) * kQ8fItemSlots;
    L.table = off;
    off += 4 * kMaxBpp;
    L.qbuf = align_up(off, 128);
    off = L.qbuf + kQ8fItemSlots * G * kQ8fD * 4;
    L.mscr = align_up(off, 16);
    off = L.mscr + 2 * kQ8fWarps * G * kQ8fD * 4;
    L.mml = off;
    off += 2 * kQ8fWarps * G * 2 * 4;
    L.stages = align_up(off, 128);
    off = L.stages + S * 2 * q8_page_bytes(BS, kQ8fD);
    L.total = off + 128;  // slack to align the dynamic shared memory base
    return L;
}

__device__ inline float q8f_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ inline float f16_bits_to_float(uint32_t h) { return __half2float(__ushort_as_half(static_cast<uint16_t>(h))); }

// acc += <q pair halves, code pair> for E4M3: two fp16 products, fp32 accumulate.
__device__ inline void fma2_f16(float &acc, uint32_t qh2, uint32_t ch2) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(qh2), "r"(ch2));
}

__device__ inline uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two_codes)));
    return h2;
}

// Self-checks (compiled in with PA_SELF_CHECK): an index or address outside
// its buffer sets bit (8 + code) of the error word and the access is skipped.
#ifdef PA_SELF_CHECK
__device__ inline bool q8f_ok(const DecodeParams &p, bool cond, int code) {
    if (!cond && p.err)
        atomicOr(p.err, 0x100u << code);
    return cond;
}
#define Q8F_OK(cond, code) q8f_ok(p, (cond), (code))
#else
#define Q8F_OK(cond, code) true
#endif

// Shared-memory loads at 32-bit shared-window addresses.
__device__ inline uint4 lds128(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
__device__ inline uint2 lds64(uint32_t a) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}
__device__ inline uint32_t lds32(uint32_t a) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
    return r;
}
__device__ inline float ldsf(uint32_t a) { return __uint_as_float(lds32(a)); }

// Query elements j .. j + 15 (j a multiple of 16) of a row held in shared
// memory as fp32, fp16 or bf16, widened to fp32 (16-byte loads).
__device__ inline void load_q16(const char *qr, int dtype, int j, float *f) {
    if (dtype == PA_F32) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 v = ld_shared_v4(qr + (j + 4 * k) * 4);
            f[4 * k] = __uint_as_float(v.x), f[4 * k + 1] = __uint_as_float(v.y);
            f[4 * k + 2] = __uint_as_float(v.z), f[4 * k + 3] = __uint_as_float(v.w);
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint4 v = ld_shared_v4(qr + (j + 8 * k) * 2);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (dtype == PA_F16) {
                const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&w[u]));
                f[8 * k + 2 * u] = h.x, f[8 * k + 2 * u + 1] = h.y;
            } else {
                f[8 * k + 2 * u] = __uint_as_float(w[u] << 16);
                f[8 * k + 2 * u + 1] = __uint_as_float(w[u] & 0xffff0000u);
            }
        }
    }
}

// The G words (4 codes each) of this lane's PV dims in one token row.
template <int G> __device__ inline void lds_pv(uint32_t a, uint32_t *w) {
    if (G == 1) {
        w[0] = lds32(a);
    } else if (G == 2) {
        const uint2 v = lds64(a);
        w[0] = v.x, w[G > 1 ? 1 : 0] = v.y;
    } else {
        const uint4 v = lds128(a);
        w[0] = v.x, w[G > 1 ? 1 : 0] = v.y, w[G > 2 ? 2 : 0] = v.z, w[G > 3 ? 3 : 0] = v.w;
    }
}

// ---------------------------------------------------------------------------

template <int G, int BS>
__device__ inline void q8f_producer(const DecodeParams &p, char *smem, const Q8fLayout &L) {
    using C = Q8fCfg<G, BS>;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    int *valid = reinterpret_cast<int *>(smem + L.valid);
    Q8fItem *items = reinterpret_cast<Q8fItem *>(smem + L.items);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + L.table);
    char *qbuf = smem + L.qbuf;
    char *stage_buf = smem + L.stages;
    const char *qg = static_cast<const char *>(p.q);
    const char *kc = static_cast<const char *>(p.k_cache);
    const char *vc = static_cast<const char *>(p.v_cache);
    const uint32_t qrow = kQ8fD * (p.q_dtype == PA_F32 ? 4 : 2);
    const uint64_t policy = policy_evict_first();

    int chunk_base = 0;
    long long chunk_prefix = 0;
    int my_len = 0, my_start = 0, my_np = 0, my_incl = 0, chunk_total = 0;
    bool chunk_ready = false;
    uint32_t t = 0;       // stages issued
    int pstage = 0;       // t % S
    uint32_t pphase = 0;  // (t / S) & 1
    int k = 0;            // items issued
    bool ok = true;
    const long long hkv = p.num_kv_heads;

    for (long long w = blockIdx.x;; w += gridDim.x) {
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
                my_np = sq < p.num_seqs ? seq_span(my_len, p.max_len, p.window, BS, p.bpp, my_start).nparts : 0;
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

        const int slot = k % kQ8fItemSlots;
        if (!mbar_wait_bounded(&iempty[slot], ((k / kQ8fItemSlots) & 1) ^ 1)) {
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
            Q8fItem it;
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
                mbar_arrive_expect_tx(&ifull[slot], G * qrow);
                bulk_g2s(qbuf + slot * G * C::kQRow, qg + (static_cast<long long>(s) * p.num_heads + kvh * G) * qrow,
                         G * qrow, &ifull[slot]);
            } else {
                mbar_arrive(&ifull[slot]);
            }
        }
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
        for (int j = 0; j < nb; ++j, ++t) {
            if (!mbar_wait_bounded(&empty[pstage], pphase ^ 1u)) {
                ok = false;
                break;
            }
            const int stage = pstage;
            if (++pstage == S) {
                pstage = 0;
                pphase ^= 1u;
            }
            if (lane == 0) {
                const int pb = tbl[j];
                valid[stage] = pb >= 0;
                if (pb >= 0 && Q8F_OK(stage >= 0 && stage < S, 0) &&
                    Q8F_OK(static_cast<long long>(pb) * p.num_kv_heads + kvh <
                               static_cast<long long>(p.num_blocks) * p.num_kv_heads, 1)) {
                    mbar_arrive_expect_tx(&full[stage], 2 * C::kPage);
                    char *dk = stage_buf + static_cast<size_t>(stage) * 2 * C::kPage;
                    const long long z = static_cast<long long>(pb) * p.num_kv_heads + kvh;
                    bulk_g2s_hint(dk, kc + z * C::kPage, C::kPage, &full[stage], policy);
                    bulk_g2s_hint(dk + C::kPage, vc + z * C::kPage, C::kPage, &full[stage], policy);
                } else {
                    mbar_arrive(&full[stage]);
                }
            }
            __syncwarp();
        }
        if (!ok)
            break;
        ++k;
    }
    if (!ok && lane == 0) {
        if (p.err)
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
        const uint32_t first = t > static_cast<uint32_t>(S) ? t - S : 0;
        for (uint32_t u = first; u < t; ++u)
            (void)mbar_wait_bounded(&full[u % S], (u / S) & 1u);
    }
    __syncwarp();
}

template <int Fmt, int G, int BS>
__device__ inline void q8f_consumer(const DecodeParams &p, char *smem, const Q8fLayout &L) {
    using C = Q8fCfg<G, BS>;
    constexpr int kW = C::kW, kTpr = C::kTpr, kP = C::kP, kR = C::kRounds, kCpl = C::kCpl, kQp = C::kQp;
    constexpr int kDG = C::kDG;
    constexpr bool kI8 = (Fmt == kFmtI8);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane / kW;         // this lane's query head within the kv head's group
    const int wl = lane % kW;        // lane within the head group
    const int gbase = lane & ~(kW - 1);
    // QK lanes: part in the low bits, so each 8-lane phase of a 128-bit shared
    // load covers 8 distinct 16-byte chunk positions of the rows it reads
    const int tok = wl / kP;         // QK: token of the round
    const int part = wl % kP;        // QK: share of the row
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
    uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
    uint64_t *mfull = reinterpret_cast<uint64_t *>(smem + L.mfull);
    uint64_t *mempty = reinterpret_cast<uint64_t *>(smem + L.mempty);
    const int *valid = reinterpret_cast<const int *>(smem + L.valid);
    const Q8fItem *items = reinterpret_cast<const Q8fItem *>(smem + L.items);
    const char *qbuf = smem + L.qbuf;
    float *mscr = reinterpret_cast<float *>(smem + L.mscr);  // [2][warps][G][D]
    float *mml = reinterpret_cast<float *>(smem + L.mml);    // [2][warps][G][2]
    const uint32_t stages_a = smem_addr(smem + L.stages);
    const int qelt = p.q_dtype == PA_F32 ? 4 : 2;

    // per-lane offsets inside a page: QK chunk i of row `tok` is the lane's
    // chunk (i + tok) mod kCpl (the rotation spreads a warp's loads over all
    // banks); PV reads this lane's dims of a row
    uint32_t qk_off[kCpl];
#pragma unroll
    for (int i = 0; i < kCpl; ++i)
        qk_off[i] = static_cast<uint32_t>(tok * 128 + (part * kCpl + (i + tok) % kCpl) * 16);
    const uint32_t pv_off = static_cast<uint32_t>(wl * kDG);

    uint32_t qp[kQp];  // query pairs of this lane's QK dims: int16x2 (INT8) or f16x2 (E4M3)
    float cq = 0.f;    // score factor (query scale * scale * log2 e)
    bool ok = true;
    for (int k = 0;; ++k) {
        const int slot = k % kQ8fItemSlots;
        if (!mbar_wait_bounded(&ifull[slot], (k / kQ8fItemSlots) & 1)) {
            ok = false;
            break;
        }
        const Q8fItem it = items[slot];
        if (it.end)
            break;
        if (it.nb > 0) {
            const char *qr = qbuf + slot * G * C::kQRow + g * kQ8fD * qelt;
            (void)Q8F_OK(slot >= 0 && slot < kQ8fItemSlots && it.s >= 0 && it.s < p.num_seqs &&
                             it.part >= 0 && it.part < p.max_parts, 9);
            // the row's largest magnitude: this lane's QK dims, then over the
            // parts of its token (they cover the row once)
            float amax = 0.f;
#pragma unroll
            for (int c = 0; c < kCpl; ++c) {
                float f[16];
                load_q16(qr, p.q_dtype, part * (kQ8fD / kP) + c * 16, f);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    amax = fmaxf(amax, fabsf(f[e]));
            }
#pragma unroll
            for (int o = 1; o < kP; o <<= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            // a row whose largest element is below 1e-30 is read as zero
            if (!(amax > 1e-30f))
                amax = 0.f;
            // query pairs in the rotated chunk order: pair 8 i + u holds dims
            // 2u, 2u + 1 of the lane's chunk (i + tok) mod kCpl
            float inv, up = 1.f;
            if (kI8) {
                // int16 query: q ~ sq * qi, sq = max|q| / 32767
                inv = amax > 0.f ? 32767.f / amax : 0.f;
                cq = amax * (1.f / 32767.f) * p.scale_log2;
            } else {
                // fp16 query scaled by 2^e so that max |q| * 2^e lies in [2^14, 2^15)
                const int e2 = amax > 0.f ? min(126, 14 - ilogbf(amax)) : 0;
                up = ldexpf(1.f, e2);
                cq = ldexpf(p.scale_log2, -e2);
                inv = 0.f;
            }
#pragma unroll
            for (int i = 0; i < kCpl; ++i) {
                float f[16];
                load_q16(qr, p.q_dtype, part * (kQ8fD / kP) + ((i + tok) % kCpl) * 16, f);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (kI8) {
                        const int a = max(-32767, min(32767, __float2int_rn(f[2 * u] * inv)));
                        const int b = max(-32767, min(32767, __float2int_rn(f[2 * u + 1] * inv)));
                        qp[i * 8 + u] = (static_cast<uint32_t>(a) & 0xffffu) | (static_cast<uint32_t>(b) << 16);
                    } else {
                        const __half2 h = __floats2half2_rn(f[2 * u] * up, f[2 * u + 1] * up);
                        qp[i * 8 + u] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&iempty[slot]);

        float m = -INFINITY, l = 0.f;
        float acc[kDG];
#pragma unroll
        for (int i = 0; i < kDG; ++i)
            acc[i] = 0.f;

        int j = (warp - it.t_first % kQ8fWarps + kQ8fWarps) % kQ8fWarps;
        const uint32_t t0 = static_cast<uint32_t>(it.t_first + j);
        int stage = static_cast<int>(t0 % S);
        uint32_t phase = (t0 / S) & 1u;
        for (; j < it.nb; j += kQ8fWarps) {
            if (!mbar_wait_bounded(&full[stage], phase)) {
                ok = false;
                break;
            }
            if (valid[stage] && Q8F_OK(stage >= 0 && stage < S, 3)) {
                const uint32_t kt = stages_a + static_cast<uint32_t>(stage) * 2 * C::kPage;
                const uint32_t vt = kt + C::kPage;
                const uint32_t sk = kt + BS * 128;  // the pages' scale rows
                const uint32_t sv = vt + BS * 128;
                const int blk = it.blk_lo + j;
                const int lo = max(it.tok_lo - blk * BS, 0);
                const int hi = min(it.tok_hi - blk * BS, BS);

                // ---- scores of the block's tokens (this lane's head)
                float sc[kR];
#pragma unroll
                for (int rd = 0; rd < kR; ++rd) {
                    const int r = rd * kTpr + tok;
                    const uint32_t rowa = kt + rd * kTpr * 128;
                    float x;
                    if (kI8) {
                        int a[4] = {0, 0, 0, 0};
#pragma unroll
                        for (int i = 0; i < kCpl; ++i) {
                            const uint32_t qa = rowa + qk_off[i];
                            const uint4 w = Q8F_OK(qa >= kt && qa + 16 <= kt + BS * 128 && (qa & 15) == 0, 4)
                                                ? lds128(qa) : make_uint4(0, 0, 0, 0);
                            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                a[u] = __dp2a_lo(static_cast<int>(qp[i * 8 + 2 * u]), static_cast<int>(ws[u]), a[u]);
                                a[u] = __dp2a_hi(static_cast<int>(qp[i * 8 + 2 * u + 1]), static_cast<int>(ws[u]), a[u]);
                            }
                        }
                        int sum = (a[0] + a[1]) + (a[2] + a[3]);
#pragma unroll
                        for (int o = 1; o < kP; o <<= 1)
                            sum += __shfl_xor_sync(0xffffffffu, sum, o);
                        x = static_cast<float>(sum);
                    } else {
                        float xa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int i = 0; i < kCpl; ++i) {
                            const uint4 w = lds128(rowa + qk_off[i]);
                            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                fma2_f16(xa[u], qp[i * 8 + 2 * u], e4m3x2_to_f16x2(ws[u] & 0xffffu));
                                fma2_f16(xa[u], qp[i * 8 + 2 * u + 1], e4m3x2_to_f16x2(ws[u] >> 16));
                            }
                        }
                        x = (xa[0] + xa[1]) + (xa[2] + xa[3]);
#pragma unroll
                        for (int o = 1; o < kP; o <<= 1)
                            x += __shfl_xor_sync(0xffffffffu, x, o);
                    }
                    const float skr = Q8F_OK(r >= 0 && r < BS, 6) ? ldsf(sk + r * 4) : 0.f;
                    sc[rd] = (r >= lo && r < hi) ? x * (cq * skr) : -INFINITY;
                }

                // ---- one running-max update per block; weights
                float mb = sc[0];
#pragma unroll
                for (int rd = 1; rd < kR; ++rd)
                    mb = fmaxf(mb, sc[rd]);
#pragma unroll
                for (int o = kP; o < kW; o <<= 1)
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
                if (mb > m) {
                    const float alpha = q8f_exp2(m - mb);
                    l *= alpha;
#pragma unroll
                    for (int i = 0; i < kDG; ++i)
                        acc[i] *= alpha;
                    m = mb;
                }
                float pw[kR];
#pragma unroll
                for (int rd = 0; rd < kR; ++rd) {
                    const float pr = q8f_exp2(sc[rd] - m);
                    l += pr;
                    pw[rd] = pr * (Q8F_OK(rd * kTpr + tok < BS, 6) ? ldsf(sv + (rd * kTpr + tok) * 4) : 0.f);
                }

                // ---- P V: this lane's kDG dims of its head
                if (kI8) {
                    // rows outside [lo, hi) have weight 0 and so quantised weight 0: the
                    // integer products ignore whatever those rows hold
                    float pm = pw[0];
#pragma unroll
                    for (int rd = 1; rd < kR; ++rd)
                        pm = fmaxf(pm, pw[rd]);
#pragma unroll
                    for (int o = kP; o < kW; o <<= 1)
                        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, o));
                    const float inv = pm > 0.f ? __fdividef(32767.f, pm) : 0.f;
                    const float ps = pm * (1.f / 32767.f);
                    uint32_t pk[kR];
#pragma unroll
                    for (int rd = 0; rd < kR; ++rd) {
                        const int pi = min(32767, __float2int_rn(pw[rd] * inv));
                        const int nb_pi = __shfl_xor_sync(0xffffffffu, pi, kP);  // the next token's lane
                        pk[rd] = (static_cast<uint32_t>(pi) & 0xffffu) | (static_cast<uint32_t>(nb_pi) << 16);
                    }
                    int ai[kDG];
#pragma unroll
                    for (int i = 0; i < kDG; ++i)
                        ai[i] = 0;
#pragma unroll
                    for (int rd = 0; rd < kR; ++rd) {
#pragma unroll
                        for (int tp = 0; tp < kTpr; tp += 2) {
                            const int ta = rd * kTpr + tp;  // the pair (ta, ta + 1)
                            const int pp = static_cast<int>(__shfl_sync(0xffffffffu, pk[rd], gbase + tp * kP));
                            uint32_t w0[G], w1[G];
                            const uint32_t a0 = vt + ta * 128 + pv_off;
                            const uint32_t a1 = vt + (ta + 1) * 128 + pv_off;
                            if (Q8F_OK(a0 >= vt && a1 + 4 * G <= vt + BS * 128 && (a0 & (4 * G - 1)) == 0 &&
                                           (a1 & (4 * G - 1)) == 0, 5)) {
                                lds_pv<G>(a0, w0);
                                lds_pv<G>(a1, w1);
                            } else {
#pragma unroll
                                for (int q4 = 0; q4 < G; ++q4)
                                    w0[q4] = w1[q4] = 0;
                            }
#pragma unroll
                            for (int q4 = 0; q4 < G; ++q4) {
                                const int xl = static_cast<int>(__byte_perm(w0[q4], w1[q4], 0x5140));
                                const int xh = static_cast<int>(__byte_perm(w0[q4], w1[q4], 0x7362));
                                ai[4 * q4 + 0] = __dp2a_lo(pp, xl, ai[4 * q4 + 0]);
                                ai[4 * q4 + 1] = __dp2a_hi(pp, xl, ai[4 * q4 + 1]);
                                ai[4 * q4 + 2] = __dp2a_lo(pp, xh, ai[4 * q4 + 2]);
                                ai[4 * q4 + 3] = __dp2a_hi(pp, xh, ai[4 * q4 + 3]);
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kDG; ++i)
                        acc[i] = fmaf(ps, static_cast<float>(ai[i]), acc[i]);
                } else {
                    // fp32 products: rows outside [lo, hi) are skipped (they may hold any bits)
#pragma unroll
                    for (int rd = 0; rd < kR; ++rd) {
#pragma unroll
                        for (int u = 0; u < kTpr; ++u) {
                            const int ta = rd * kTpr + u;
                            const float pu = __shfl_sync(0xffffffffu, pw[rd], gbase + u * kP);
                            if (ta < lo || ta >= hi)
                                continue;
                            uint32_t w[G];
                            lds_pv<G>(vt + ta * 128 + pv_off, w);
#pragma unroll
                            for (int q4 = 0; q4 < G; ++q4) {
                                const uint32_t h01 = e4m3x2_to_f16x2(w[q4] & 0xffffu);
                                const uint32_t h23 = e4m3x2_to_f16x2(w[q4] >> 16);
                                acc[4 * q4 + 0] = fmaf(pu, f16_bits_to_float(h01), acc[4 * q4 + 0]);
                                acc[4 * q4 + 1] = fmaf(pu, f16_bits_to_float(h01 >> 16), acc[4 * q4 + 1]);
                                acc[4 * q4 + 2] = fmaf(pu, f16_bits_to_float(h23), acc[4 * q4 + 2]);
                                acc[4 * q4 + 3] = fmaf(pu, f16_bits_to_float(h23 >> 16), acc[4 * q4 + 3]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
            stage += kQ8fWarps;
            if (stage >= S) {
                stage -= S;
                phase ^= 1u;
            }
        }
        if (!ok)
            break;

        // ---- merge the 4 warps' states of this item (double-buffered by item parity)
        // l holds this lane's tokens (the parts of a token hold copies): sum over tokens
#pragma unroll
        for (int o = kP; o < kW; o <<= 1)
            l += __shfl_xor_sync(0xffffffffu, l, o);
        const int b = k & 1;
        const uint32_t use = static_cast<uint32_t>(k >> 1) & 1u;
        if (!mbar_wait_bounded(&mempty[b], use ^ 1u)) {
            ok = false;
            break;
        }
        float *dst = mscr + ((b * kQ8fWarps + warp) * G + g) * kQ8fD + wl * kDG;
#pragma unroll
        for (int i = 0; i < kDG; i += 4)
            *reinterpret_cast<float4 *>(dst + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
        if (wl == 0) {
            mml[((b * kQ8fWarps + warp) * G + g) * 2] = m;
            mml[((b * kQ8fWarps + warp) * G + g) * 2 + 1] = l;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&mfull[b]);
        if (!mbar_wait_bounded(&mfull[b], use)) {
            ok = false;
            break;
        }
        for (int idx = warp * 32 + lane; idx < G * kQ8fD; idx += kQ8fWarps * 32) {
            const int gg = idx / kQ8fD, dd = idx % kQ8fD;
            float M = -INFINITY;
#pragma unroll
            for (int w2 = 0; w2 < kQ8fWarps; ++w2)
                M = fmaxf(M, mml[((b * kQ8fWarps + w2) * G + gg) * 2]);
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w2 = 0; w2 < kQ8fWarps; ++w2) {
                    const float sw = q8f_exp2(mml[((b * kQ8fWarps + w2) * G + gg) * 2] - M);
                    num = fmaf(mscr[((b * kQ8fWarps + w2) * G + gg) * kQ8fD + dd], sw, num);
                    den = fmaf(mml[((b * kQ8fWarps + w2) * G + gg) * 2 + 1], sw, den);
                }
            }
            const long long orow = static_cast<long long>(it.s) * p.num_heads + it.kvh * G + gg;
            if (!Q8F_OK(orow >= 0 && orow < static_cast<long long>(p.num_seqs) * p.num_heads, 7))
                continue;
            if (it.nparts == 1 && !p.force_partial) {
                store_out(p.out, p.out_dtype, orow * kQ8fD + dd, den > 0.f ? num / den : 0.f);
            } else {
                const long long pr = orow * p.max_parts + it.part;
                if (!Q8F_OK(p.part_acc != nullptr && it.part >= 0 && it.part < p.max_parts, 8))
                    continue;
                p.part_acc[pr * kQ8fD + dd] = num;
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

// CTAs per SM the register budget is set for: 5 for one query head per kv
// head (20 consumer warps, <= 72 registers a thread), 3 for grouped heads.
template <int G> struct Q8fOccupancy {
    static constexpr int kMinBlocks = G == 1 ? 5 : 3;
};

template <int Fmt, int G, int BS>
__global__ void __launch_bounds__(kQ8fThreads, Q8fOccupancy<G>::kMinBlocks) pa_decode_q8f_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const Q8fLayout L = q8f_smem_layout(p.stages, BS, G);
    // Stage t belongs to consumer warp t % 4.  With a stage count that is not a
    // multiple of 4, one stage would pass between warps, and a warp running a
    // full ring ahead could see its parity wait satisfied by an older phase of
    // that stage.  The host never launches such a count; refuse it here too.
    if (p.stages < kQ8fWarps || p.stages % kQ8fWarps != 0) {
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
        for (int i = 0; i < kQ8fItemSlots; ++i) {
            mbar_init(&ifull[i], 1);
            mbar_init(&iempty[i], kQ8fWarps);
        }
        uint64_t *mfull = reinterpret_cast<uint64_t *>(smem + L.mfull);
        uint64_t *mempty = reinterpret_cast<uint64_t *>(smem + L.mempty);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&mfull[i], kQ8fWarps);
            mbar_init(&mempty[i], kQ8fWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if ((threadIdx.x >> 5) == kQ8fWarps)
        q8f_producer<G, BS>(p, smem, L);
    else
        q8f_consumer<Fmt, G, BS>(p, smem, L);
}

}  // namespace pa
