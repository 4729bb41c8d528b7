// Paged decode attention over an 8-bit KV cache, head_dim 128, query groups
// G in {1, 2, 4}: the persistent, warp-specialised kernel for 8-bit pages.
//
// What it computes is pa_decode's attention with every cached element read as
// code * scale of its row (pa_quant.cuh): for token t of a sequence with codes
// c_t, c'_t and row scales sk_t, sv_t,
//   x_t = scale * sk_t * <q, c_t>,  out = sum_t e^(x_t - m) sv_t c'_t / sum_t e^(x_t - m).
//
// Work: items (sequence, group of 4 consecutive kv heads, context partition).
// A block's pages of consecutive kv heads are adjacent in the pool, so the
// producer warp moves, per block, the 4 heads' K pages with one 1-D bulk copy
// and their V pages with another (about 8.7 KB each at block size 16: copies
// of a few KB keep HBM near its copy bandwidth, where single 2 KB pages do
// not).  Consumer warp w serves kv head 4 * group + w over every block of the
// item, with its own running max, denominator and accumulator, and writes its
// rows (or partition partials) itself: no merge between warps.  Every warp
// consumes every stage (empty barriers count 4 arrivals), so the stage ring
// has no ownership constraint.
//
// Consumers: a warp is G head groups of W = 32 / G lanes; each lane serves one
// query head.  Per block of block_size tokens:
//  - QK: a head group's lanes are (token, part) pairs, part in the low lane
//    bits: kTpr tokens per round, kP lanes per token (a 128-code row split kP
//    ways).  Pages land unswizzled; the lanes of a token read its chunks in an
//    order rotated by the token index (their query pairs are stored rotated
//    the same way), so every 8-lane phase of a 16-byte shared load covers 8
//    distinct bank groups.
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
// Every wait is bounded (PA_DEVERR_TIMEOUT); table entries outside the pool
// are never dereferenced (PA_DEVERR_BAD_BLOCK).
#pragma once

#include "pa_decode.cuh"
#include "pa_quant.cuh"

#include <type_traits>

namespace pa {

constexpr int kQ8fWarps = 4;  // consumer warps = kv heads per item
constexpr int kQ8fThreads = (kQ8fWarps + 1) * 32;
constexpr int kQ8fItemSlots = 4;
constexpr int kQ8fD = 128;
constexpr int kQ8fNearBlocks = 4;  // blocks of an item still to issue when the next item is claimed
// INT8 query rows take the int16 grid while max|q| * d <= 16 * sum |q|
// (largest element at most 16 times the row's mean magnitude)
constexpr float kQ8fWideRatio = 16.f;

struct Q8fItem {
    int s, kvh0, nh, part;  // sequence, first kv head, kv heads in the item (<= 4), partition
    int nparts;
    int nb;       // blocks of the item (0: empty sequence)
    int tok_lo;   // attended tokens of the item: [tok_lo, tok_hi)
    int tok_hi;
    int blk_lo;   // first logical block
    int t_first;  // pipeline stage counter of the first block
    int end;      // 1: no more items
    int pad;
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
    static_assert(kTpr % 2 == 0 && kP >= 1 && kCpl >= 1 && BS % kTpr == 0, "lane mapping");
};

struct Q8fLayout {
    uint32_t full, empty, ifull, iempty, valid, items, table, qbuf, stages, total;
};

// Stage = [K pages of the 4 heads][V pages of the 4 heads]; qrow = bytes of one query row.
__host__ __device__ inline Q8fLayout q8f_smem_layout(int S, int BS, int G, int qrow) {
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
    L.valid = off;
    off += 4 * S;
    L.items = align_up(off, 16);
    off = L.items + sizeof(Q8fItem) * kQ8fItemSlots;
    L.table = off;
    off += 4 * kMaxBpp;
    L.qbuf = align_up(off, 128);
    off = L.qbuf + kQ8fItemSlots * kQ8fWarps * G * qrow;
    L.stages = align_up(off, 128);
    off = L.stages + S * 2 * kQ8fWarps * q8_page_bytes(BS, kQ8fD);
    L.total = off + 128;  // slack to align the dynamic shared memory base
    return L;
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

// Two of the four INT8 codes of a word as exact fp16 values: the selected
// bytes, biased to unsigned, become the low mantissa bits of 1024 (fp16
// 0x6400), and subtracting 1024 + 128 leaves the signed code.  sel 0x4140
// takes bytes 0 and 1, 0x4342 bytes 2 and 3.
__device__ inline uint32_t i8x2_to_f16x2(uint32_t four_codes, uint32_t sel) {
    const uint32_t u = __byte_perm(four_codes ^ 0x80808080u, 0x64646464u, sel);
    const __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&u), __half2half2(__ushort_as_half(0x6480u)));
    return *reinterpret_cast<const uint32_t *>(&h);
}

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
__device__ inline void q8f_producer(const DecodeParams &p, char *smem, const Q8fLayout &L, int qrow) {
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
    const uint64_t policy = policy_evict_first();
    const uint32_t stage_bytes = 2u * kQ8fWarps * C::kPage;

    ItemScan scan;
    uint32_t t = 0;       // stages issued
    int pstage = 0;       // t % S
    uint32_t pphase = 0;  // (t / S) & 1
    int k = 0;            // items issued
    bool ok = true;
    const int nquads = (p.num_kv_heads + kQ8fWarps - 1) / kQ8fWarps;

    // the next item is claimed when the current one has kQ8fNearBlocks
    // blocks left to issue: a CTA never holds a claim it is far from
    // starting, so the launch's last items go to the CTAs that run out first
    ItemClaim claim;
    claim.start();
    for (;; claim.next(p)) {
        const long long w = claim.w;
        const long long f = w / nquads;
        const int kvh0 = static_cast<int>(w % nquads) * kQ8fWarps;
        int part = 0, len = 0, start = 0;
        const int s = scan.find(p, BS, f, part, len, start);

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
        const int nh = min(kQ8fWarps, p.num_kv_heads - kvh0);
        if (lane == 0) {
            Q8fItem it;
            it.s = s;
            it.kvh0 = kvh0;
            it.nh = nh;
            it.part = part;
            it.nparts = sp.nparts;
            it.nb = nb;
            it.tok_lo = max(sp.start, blk_lo * BS);
            it.tok_hi = min(sp.end, (blk_lo + nb) * BS);
            it.blk_lo = blk_lo;
            it.t_first = static_cast<int>(t);
            it.end = 0;
            it.pad = 0;
            items[slot] = it;
            if (nb > 0) {
                // the query rows of the item's heads are consecutive in q
                const uint32_t qbytes = static_cast<uint32_t>(nh * G * qrow);
                mbar_arrive_expect_tx(&ifull[slot], qbytes);
                bulk_g2s(qbuf + slot * kQ8fWarps * G * qrow,
                         qg + (static_cast<long long>(s) * p.num_heads + kvh0 * G) * qrow, qbytes, &ifull[slot]);
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
            if (j == max(0, nb - kQ8fNearBlocks))
                claim.claim_next(p);
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
                if (pb >= 0 && Q8F_OK(stage >= 0 && stage < S, 0)) {
                    const uint32_t bytes = static_cast<uint32_t>(nh * C::kPage);
                    mbar_arrive_expect_tx(&full[stage], 2 * bytes);
                    char *dk = stage_buf + static_cast<size_t>(stage) * stage_bytes;
                    const long long z = static_cast<long long>(pb) * p.num_kv_heads + kvh0;
                    bulk_g2s_hint(dk, kc + z * C::kPage, bytes, &full[stage], policy);
                    bulk_g2s_hint(dk + kQ8fWarps * C::kPage, vc + z * C::kPage, bytes, &full[stage], policy);
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
    claim.finish(p);
    __syncwarp();
}

template <int Fmt, int G, int BS>
__device__ inline void q8f_consumer(const DecodeParams &p, char *smem, const Q8fLayout &L, int qrow) {
    using C = Q8fCfg<G, BS>;
    constexpr int kW = C::kW, kTpr = C::kTpr, kP = C::kP, kR = C::kRounds, kCpl = C::kCpl, kQp = C::kQp;
    constexpr int kDG = C::kDG;
    constexpr bool kI8 = (Fmt == kFmtI8);
    const int warp = threadIdx.x >> 5;  // kv head kvh0 + warp of each item
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
    const int *valid = reinterpret_cast<const int *>(smem + L.valid);
    const Q8fItem *items = reinterpret_cast<const Q8fItem *>(smem + L.items);
    const char *qbuf = smem + L.qbuf;
    const uint32_t stages_a = smem_addr(smem + L.stages);
    const uint32_t stage_bytes = 2u * kQ8fWarps * C::kPage;

    // per-lane offsets inside a page: QK chunk i of row `tok` is the lane's
    // chunk (i + tok) mod kCpl (the rotation spreads a warp's loads over all
    // banks); PV reads this lane's dims of a row
    uint32_t qk_off[kCpl];
#pragma unroll
    for (int i = 0; i < kCpl; ++i)
        qk_off[i] = static_cast<uint32_t>(tok * 128 + (part * kCpl + (i + tok) % kCpl) * 16);
    const uint32_t pv_off = static_cast<uint32_t>(wl * kDG);

    uint32_t qp[kQp];  // query pairs of this lane's QK dims: int16x2 (INT8) or f16x2 (E4M3, wide INT8)
    float cq = 0.f;    // score factor (query scale * scale * log2 e)
    bool wide = false; // INT8: this warp's query rows are held as fp16 (exact products), not int16
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
        const bool active = warp < it.nh;  // a head past num_kv_heads in the last group idles
        if (it.nb > 0 && active) {
            const char *qr = qbuf + (slot * kQ8fWarps + warp) * G * qrow + g * qrow;
            // the row's largest magnitude: this lane's QK dims, then over the
            // parts of its token (they cover the row once)
            float amax = 0.f, sabs = 0.f;
#pragma unroll
            for (int c = 0; c < kCpl; ++c) {
                float f[16];
                load_q16(qr, p.q_dtype, part * (kQ8fD / kP) + c * 16, f);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    amax = fmaxf(amax, fabsf(f[e]));
                    if (kI8)
                        sabs += fabsf(f[e]);
                }
            }
#pragma unroll
            for (int o = 1; o < kP; o <<= 1) {
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                if (kI8)
                    sabs += __shfl_xor_sync(0xffffffffu, sabs, o);
            }
            // a row whose largest element is below 1e-30 is read as zero
            if (!(amax > 1e-30f))
                amax = 0.f;
            if (kI8) {
                // the int16 grid (step max|q| / 32767) keeps every element to
                // within 2^-11 of the row's mean magnitude when max|q| <= 16
                // mean|q|; a warp holding a row of wider range (a few outlier
                // elements) takes fp16 products instead, for all of its rows
                // (exact for fp16 and bf16 queries, as for E4M3 codes)
                wide = __any_sync(0xffffffffu, amax * static_cast<float>(kQ8fD) > kQ8fWideRatio * sabs);
            }
            // query pairs in the rotated chunk order: pair 8 i + u holds dims
            // 2u, 2u + 1 of the lane's chunk (i + tok) mod kCpl
            float inv, up = 1.f;
            if (kI8 && !wide) {
                // int16 query: q ~ sq * qi, sq = max|q| / 32767
                inv = amax > 0.f ? 32767.f / amax : 0.f;
                cq = amax * (1.f / 32767.f) * p.scale_log2;
            } else {
                // fp16 query (E4M3, or INT8 of wide range) scaled by 2^e so that
                // max |q| * 2^e lies in [2^14, 2^15)
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
                    if (kI8 && !wide) {
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

        const uint32_t t0 = static_cast<uint32_t>(it.t_first);
        int stage = static_cast<int>(t0 % S);
        uint32_t phase = (t0 / S) & 1u;
        // the block loop, compiled twice: int16 query products (kExact false)
        // and, for a warp whose INT8 rows are of wide range, fp16 products
        auto blocks = [&](auto exact_tag) {
            constexpr bool kExact = decltype(exact_tag)::value;
            for (int j = 0; j < it.nb; ++j) {
                if (!mbar_wait_bounded(&full[stage], phase)) {
                    ok = false;
                    break;
                }
                if (active && valid[stage] && Q8F_OK(stage >= 0 && stage < S, 3)) {
                    const uint32_t kt = stages_a + static_cast<uint32_t>(stage) * stage_bytes + warp * C::kPage;
                    const uint32_t vt = kt + kQ8fWarps * C::kPage;
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
                        if (kI8 && !kExact) {
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
                                    if (kI8) {
                                        fma2_f16(xa[u], qp[i * 8 + 2 * u], i8x2_to_f16x2(ws[u], 0x4140u));
                                        fma2_f16(xa[u], qp[i * 8 + 2 * u + 1], i8x2_to_f16x2(ws[u], 0x4342u));
                                    } else {
                                        fma2_f16(xa[u], qp[i * 8 + 2 * u], e4m3x2_to_f16x2(ws[u] & 0xffffu));
                                        fma2_f16(xa[u], qp[i * 8 + 2 * u + 1], e4m3x2_to_f16x2(ws[u] >> 16));
                                    }
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
                        pw[rd] = pr * ldsf(sv + (rd * kTpr + tok) * 4);
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
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        };
        if (kI8 && wide)
            blocks(std::true_type{});
        else
            blocks(std::false_type{});
        if (!ok)
            break;

        // ---- this warp's head: the output rows, or the partition's partials
        if (active) {
            // l holds this lane's tokens (the parts of a token hold copies): sum over tokens
#pragma unroll
            for (int o = kP; o < kW; o <<= 1)
                l += __shfl_xor_sync(0xffffffffu, l, o);
            const long long orow = static_cast<long long>(it.s) * p.num_heads + (it.kvh0 + warp) * G + g;
            if (Q8F_OK(orow >= 0 && orow < static_cast<long long>(p.num_seqs) * p.num_heads, 7)) {
                if (it.nparts == 1 && !p.force_partial) {
                    const float rl = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                    for (int i = 0; i < kDG; ++i)
                        store_out(p.out, p.out_dtype, orow * kQ8fD + wl * kDG + i, acc[i] * rl);
                } else if (Q8F_OK(p.part_acc != nullptr && it.part >= 0 && it.part < p.max_parts, 8)) {
                    const long long pr = orow * p.max_parts + it.part;
                    float *dst = p.part_acc + pr * kQ8fD + wl * kDG;
#pragma unroll
                    for (int i = 0; i < kDG; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
                    if (wl == 0) {
                        p.part_ml[pr * 2] = m;
                        p.part_ml[pr * 2 + 1] = l;
                    }
                }
            }
        }
    }
    if (!ok && lane == 0 && p.err)
        atomicOr(p.err, PA_DEVERR_TIMEOUT);
}

// CTAs per SM the register budget is set for: 5 for one query head per kv
// head (<= 72 registers a thread), 3 for grouped heads.
template <int G> struct Q8fOccupancy {
    static constexpr int kMinBlocks = G == 1 ? 5 : 3;
};

template <int Fmt, int G, int BS>
__global__ void __launch_bounds__(kQ8fThreads, Q8fOccupancy<G>::kMinBlocks) pa_decode_q8f_kernel(const DecodeParams p) {
    // the next kernel on the stream may be launched now (it waits for this
    // grid); this one waits for the kernel before it
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(128) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int qrow = kQ8fD * (p.q_dtype == PA_F32 ? 4 : 2);
    const Q8fLayout L = q8f_smem_layout(p.stages, BS, G, qrow);
    if (p.stages < 2) {
        if (threadIdx.x == 0 && p.err)
            atomicOr(p.err, PA_DEVERR_BAD_LAUNCH);
        return;
    }
    if (threadIdx.x == 0) {
        uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.full);
        uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.empty);
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kQ8fWarps);
        }
        uint64_t *ifull = reinterpret_cast<uint64_t *>(smem + L.ifull);
        uint64_t *iempty = reinterpret_cast<uint64_t *>(smem + L.iempty);
        for (int i = 0; i < kQ8fItemSlots; ++i) {
            mbar_init(&ifull[i], 1);
            mbar_init(&iempty[i], kQ8fWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if ((threadIdx.x >> 5) == kQ8fWarps)
        q8f_producer<G, BS>(p, smem, L, qrow);
    else
        q8f_consumer<Fmt, G, BS>(p, smem, L, qrow);
    __syncthreads();
    release_claims(p);
}

}  // namespace pa
