/*
 * Plain CPU oracle for paged decode attention, KV append and block copy.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product calls this file: only the
 * tests, the smoke check and the benchmark's CPU-baseline / reference leg load
 * the shared library built from it.  It shares no code, header or table with
 * the CUDA library; the dtype codes below are an interface agreement (the same
 * small integers the C ABI uses), re-declared here.
 *
 * Everything is written for obviousness, not speed: fp64 arithmetic, one token
 * at a time, in the order the definitions state.  Every function is pinned by
 * the CPU tests (worked example, brute force over a contiguous copy through a
 * library softmax, permutation invariance, closed forms).
 *
 * Sources (web pages on PagedAttention):
 *  - "PagedAttention: From Operating System Virtual Memory to Large Language
 *    Model Memory Systems", section 2 Background: the attention formula
 *    softmax(Q K^T / sqrt(d)) V.
 *  - "PagedAttention — 把 KV cache 当虚拟内存页来管理", 实践案例 案例 2: the
 *    block-table lookup locate(t) = (table[t / block_size], t % block_size);
 *    "attention kernel 多查一次表" (the kernel reads K/V through the table).
 *    核心要点: every generated token's key/value is saved and re-read.
 *  - "KV Cache与长上下文管理", section "让 Round Robin / Sliding Window 变成 O(1)
 *    操作": a sliding window is realised by recycling pages and rewriting the
 *    page table; the attended set is the most recent tokens.  The same page's
 *    KV-cache quantisation passage (FP16 -> INT8 -> INT4) and the mjmagnets
 *    article's section 4.1 mixed-precision pages (INT8 for rarely used pages):
 *    8-bit caches, read here as symmetric per-row quantisation (one fp32
 *    scale per cached (token, kv head) row, the codes decided in fp32).
 *
 * 8-bit cache pages.  A (block, kv head) page of an 8-bit pool holds the
 * block's block_size code rows of head_dim bytes, followed by
 * scale_rows = ceil(4 * block_size / head_dim) rows whose first
 * 4 * block_size bytes are the rows' fp32 scales (the rest zero):
 *   pool [num_blocks][num_kv_heads][block_size + scale_rows][head_dim] bytes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_I8 = 3, ORC_E4M3 = 4 };

/* ------------------------------------------------------------------ */
/* Exact element conversions (every fp16/bf16/fp32 value is a double). */

static double orc_f16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* subnormal or zero */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25);  /* 1.mant * 2^(e-15) */
    return sign ? -v : v;
}

static double orc_bf16_bits_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;                 /* bf16 = top half of fp32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double orc_load(const void *base, int dtype, int64_t index)
{
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * index, 4);
        return (double)f;
    }
    uint16_t u;
    memcpy(&u, (const char *)base + 2 * index, 2);
    return dtype == ORC_F16 ? orc_f16_bits_to_double(u) : orc_bf16_bits_to_double(u);
}

double orc_element_to_double(const void *base, int dtype, int64_t index)
{
    return orc_load(base, dtype, index);
}

/* ------------------------------------------------------------------ */
/* 8-bit codes.
 *
 * INT8: two's-complement byte, value = code.
 * E4M3 (the OCP 8-bit floating-point format, E4M3 variant): sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes the
 * subnormals m/8 * 2^-6; there are no infinities, S.1111.111 is NaN, so the
 * largest finite value is 1.75 * 2^8 = 448.
 */
static double orc_i8_to_double(uint8_t c)
{
    return (double)(c < 128 ? (int)c : (int)c - 256);
}

static double orc_e4m3_to_double(uint8_t c)
{
    const int sign = c >> 7, expo = (c >> 3) & 15, mant = c & 7;
    double v;
    if (expo == 15 && mant == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)mant, -9);              /* m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + mant), expo - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

double orc_code_to_double(uint8_t code, int fmt)
{
    return fmt == ORC_I8 ? orc_i8_to_double(code) : orc_e4m3_to_double(code);
}

/* Nearest E4M3 value to a finite float, ties to the even mantissa; finite
 * values beyond 448 saturate to +-448.  The sign of zero is kept. */
static uint8_t orc_e4m3_from_float(float f)
{
    const uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0)
        return sign | 0x7e;                       /* 1.75 * 2^8 */
    /* a lies in [2^b, 2^(b+1)); below 2^-6 the subnormals share the spacing
     * of the lowest binade.  Spacing of representable values: 2^(b-3). */
    int e2;
    (void)frexp(a, &e2);                          /* a = f * 2^e2, f in [0.5, 1) */
    int b = a > 0.0 ? e2 - 1 : -6;
    if (b < -6)
        b = -6;
    const double quantum = ldexp(1.0, b - 3);
    const double r = nearbyint(a / quantum);      /* exact division; ties to even */
    const double v = r * quantum;                 /* at most 448 here */
    if (v == 0.0)
        return sign;
    (void)frexp(v, &e2);
    const int bv = e2 - 1;
    if (bv < -6)                                  /* subnormal: v = m * 2^-9 */
        return sign | (uint8_t)(int)ldexp(v, 9);
    const int m = (int)ldexp(v, 3 - bv) - 8;      /* 1.mmm -> mmm */
    return sign | (uint8_t)((bv + 7) << 3) | (uint8_t)m;
}

uint8_t orc_e4m3_encode(float f)
{
    return orc_e4m3_from_float(f);
}

/* Quantise one row of d elements (row `row` of x, dtype in_dtype):
 *   amax  = max |x_j|                      (exact: every input is an fp32 value)
 *   scale = amax / Q in fp32, Q = 127 (INT8) or 448 (E4M3)
 *   code_j = INT8: round-half-even(x_j / scale) clamped to [-127, 127]
 *            E4M3: nearest E4M3 value to x_j / scale (the quotient rounded
 *                  to fp32 first, then to E4M3)
 * A row of zeros gets scale 0 and zero codes.  Dequantised value:
 * code_j * scale (exact in fp64). */
static void orc_quantize_row(const void *x, int in_dtype, int64_t row, int d, int fmt, uint8_t *codes,
                             float *scale)
{
    const int64_t first = row * d;
    float amax = 0.0f;
    for (int j = 0; j < d; ++j) {
        const float a = fabsf((float)orc_load(x, in_dtype, first + j));
        if (a > amax)
            amax = a;
    }
    const float q = fmt == ORC_I8 ? 127.0f : 448.0f;
    const float s = amax / q;
    *scale = s;
    for (int j = 0; j < d; ++j) {
        if (s == 0.0f) {
            codes[j] = 0;
            continue;
        }
        const float v = (float)orc_load(x, in_dtype, first + j) / s;
        if (fmt == ORC_I8) {
            float r = rintf(v);
            if (r > 127.0f)
                r = 127.0f;
            if (r < -127.0f)
                r = -127.0f;
            const int c = (int)r;
            codes[j] = (uint8_t)(c < 0 ? c + 256 : c);
        } else {
            codes[j] = orc_e4m3_from_float(v);
        }
    }
}

/* Quantise num_rows rows of d elements: codes [num_rows][d], scales [num_rows].
 * Returns 0, or -4 for a bad format / dtype. */
int orc_quantize_rows(const void *x, int in_dtype, int64_t num_rows, int d, int fmt, uint8_t *codes,
                      float *scales)
{
    if ((fmt != ORC_I8 && fmt != ORC_E4M3) || (in_dtype != ORC_F32 && in_dtype != ORC_F16 &&
                                               in_dtype != ORC_BF16) || d <= 0)
        return -4;
    for (int64_t r = 0; r < num_rows; ++r)
        orc_quantize_row(x, in_dtype, r, d, fmt, codes + r * d, &scales[r]);
    return 0;
}

int orc_scale_rows(int block_size, int head_dim)
{
    return (4 * block_size + head_dim - 1) / head_dim;
}

/* Value of cache element `elem` (index into [num_blocks][H_kv][bs][d], the
 * logical element order): the element itself for fp32/fp16/bf16 caches; for
 * 8-bit pages, code * scale of its row, both read from the row's page. */
static double orc_cache_value(const void *cache, int cache_dtype, int64_t elem, int d, int bs)
{
    if (cache_dtype == ORC_I8 || cache_dtype == ORC_E4M3) {
        const int64_t row = elem / d;                 /* (page, r) */
        const int64_t page = row / bs;
        const int64_t r = row % bs;
        const int64_t page_bytes = (int64_t)(bs + orc_scale_rows(bs, d)) * d;
        const uint8_t *pg = (const uint8_t *)cache + page * page_bytes;
        float sc;
        memcpy(&sc, pg + (int64_t)bs * d + 4 * r, 4);
        return orc_code_to_double(pg[r * d + elem % d], cache_dtype) * (double)sc;
    }
    return orc_load(cache, cache_dtype, elem);
}

/* ------------------------------------------------------------------ */
/* Address translation (案例 2): logical token -> (physical block, offset). */

int orc_locate(const int32_t *block_table, int table_len, int block_size,
               int64_t token, int32_t *physical, int32_t *offset)
{
    if (block_size <= 0 || token < 0)
        return -1;
    int64_t logical = token / block_size;
    if (logical >= table_len)
        return -1;
    *physical = block_table[logical];
    *offset = (int32_t)(token % block_size);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Paged decode attention for one (sequence, query head).
 *
 * Cache layout (the pages fix none; this is the interface the library uses):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *   q                : [num_seqs][num_heads][head_dim]
 *   block_tables     : int32 [num_seqs][max_blocks_per_seq]
 * Query head h reads kv head h / (num_heads / num_kv_heads).
 * Attended tokens: [start, L) with start = max(0, L - window) when window > 0.
 *
 * invalid_policy: 0 -> an out-of-range physical block id is an error (-2);
 *                 1 -> tokens in such blocks are left out of the softmax and
 *                      *skipped is incremented (the library's documented
 *                      behaviour for bad table contents).
 * Output: out_row[head_dim]; zeros when no token is attended.
 */
typedef struct {
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size;
    double scale;
    int window, dtype, max_blocks_per_seq, num_blocks, invalid_policy;
    int cache_dtype;                /* element type of k_cache / v_cache (8-bit: pages) */
} orc_args;

static int orc_one(const orc_args *a, int s, int h, double *out_row, int64_t *skipped)
{
    const int d = a->head_dim;
    const int group = a->num_heads / a->num_kv_heads;
    const int kvh = h / group;
    const int64_t L = a->context_lens[s];
    int64_t start = 0;
    if (a->window > 0 && L > a->window)
        start = L - a->window;

    for (int j = 0; j < d; ++j)
        out_row[j] = 0.0;
    if (L <= 0)
        return 0;

    const int64_t n = L - start;
    double *x = (double *)malloc(sizeof(double) * (size_t)n);   /* scores */
    int64_t *row = (int64_t *)malloc(sizeof(int64_t) * (size_t)n); /* cache row of token, -1 if skipped */
    if (!x || !row) {
        free(x);
        free(row);
        return -3;
    }

    const int64_t q_base = ((int64_t)s * a->num_heads + h) * d;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t t = start + i;
        int32_t phys, off;
        if (orc_locate(a->block_tables + (int64_t)s * a->max_blocks_per_seq,
                       a->max_blocks_per_seq, a->block_size, t, &phys, &off) != 0) {
            free(x);
            free(row);
            return -1;
        }
        if (phys < 0 || phys >= a->num_blocks) {
            if (a->invalid_policy == 0) {
                free(x);
                free(row);
                return -2;
            }
            row[i] = -1;
            ++*skipped;
            continue;
        }
        /* element index of k_t[0] in [num_blocks][num_kv_heads][block_size][head_dim] */
        row[i] = (((int64_t)phys * a->num_kv_heads + kvh) * a->block_size + off) * d;
        double dot = 0.0;
        for (int j = 0; j < d; ++j)
            dot += orc_load(a->q, a->dtype, q_base + j) *
                   orc_cache_value(a->k_cache, a->cache_dtype, row[i] + j, d, a->block_size);
        x[i] = a->scale * dot;
    }

    /* softmax over the attended tokens, then the weighted mean of V */
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
        if (row[i] >= 0 && x[i] > m)
            m = x[i];
    if (m == -INFINITY) {           /* every token skipped: output stays zero */
        free(x);
        free(row);
        return 0;
    }
    double denom = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (row[i] < 0)
            continue;
        const double w = exp(x[i] - m);
        denom += w;
        for (int j = 0; j < d; ++j)
            out_row[j] += w * orc_cache_value(a->v_cache, a->cache_dtype, row[i] + j, d, a->block_size);
    }
    for (int j = 0; j < d; ++j)
        out_row[j] /= denom;

    free(x);
    free(row);
    return 0;
}

typedef struct {
    const orc_args *a;
    const int32_t *pairs; /* (s, h) pairs or NULL for all */
    int64_t num_items, first, stride;
    double *out;
    int status;
    int64_t skipped;
} orc_job;

static void *orc_worker(void *p)
{
    orc_job *job = (orc_job *)p;
    const orc_args *a = job->a;
    for (int64_t it = job->first; it < job->num_items; it += job->stride) {
        int s, h;
        if (job->pairs) {
            s = job->pairs[2 * it];
            h = job->pairs[2 * it + 1];
        } else {
            s = (int)(it / a->num_heads);
            h = (int)(it % a->num_heads);
        }
        int rc = orc_one(a, s, h, job->out + it * a->head_dim, &job->skipped);
        if (rc != 0 && job->status == 0)
            job->status = rc;
    }
    return NULL;
}

/*
 * out: fp64 [num_pairs][head_dim] when pairs != NULL (pairs = int32 (s, h)
 * list), else [num_seqs][num_heads][head_dim].  The outer (s, h) loop is split
 * across num_threads threads; the per-(s, h) code is the same either way.
 * Returns 0, or a negative error; *skipped_out (nullable) receives the number
 * of tokens left out under invalid_policy 1.
 */
/* Same, for a cache of cache_dtype (fp32/fp16/bf16, or 8-bit pages) and
 * queries of q_dtype. */
int orc_paged_attention_cache(double *out, const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *context_lens,
                              int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int block_size, double scale, int window, int q_dtype, int cache_dtype,
                              int max_blocks_per_seq, int num_blocks, int invalid_policy,
                              const int32_t *pairs, int64_t num_pairs, int num_threads,
                              int64_t *skipped_out)
{
    const int quant = cache_dtype == ORC_I8 || cache_dtype == ORC_E4M3;
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || (q_dtype != ORC_F32 && q_dtype != ORC_F16 && q_dtype != ORC_BF16) ||
        (!quant && cache_dtype != ORC_F32 && cache_dtype != ORC_F16 && cache_dtype != ORC_BF16))
        return -4;
    orc_args a = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                  num_kv_heads, head_dim, block_size, scale, window, q_dtype,
                  max_blocks_per_seq, num_blocks, invalid_policy, cache_dtype};
    const int64_t items = pairs ? num_pairs : (int64_t)num_seqs * num_heads;
    if (pairs)
        for (int64_t i = 0; i < num_pairs; ++i)
            if (pairs[2 * i] < 0 || pairs[2 * i] >= num_seqs || pairs[2 * i + 1] < 0 ||
                pairs[2 * i + 1] >= num_heads)
                return -4;
    if (num_threads < 1)
        num_threads = 1;
    if (num_threads > 256)
        num_threads = 256;
    orc_job jobs[256];
    pthread_t tids[256];
    for (int t = 0; t < num_threads; ++t) {
        jobs[t] = (orc_job){&a, pairs, items, t, num_threads, out, 0, 0};
    }
    int started = 0;
    for (int t = 1; t < num_threads; ++t) {
        if (pthread_create(&tids[t], NULL, orc_worker, &jobs[t]) != 0)
            break;
        started = t;
    }
    orc_worker(&jobs[0]);
    /* threads that failed to start: run their share here */
    for (int t = started + 1; t < num_threads; ++t)
        orc_worker(&jobs[t]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tids[t], NULL);
    int status = 0;
    int64_t skipped = 0;
    for (int t = 0; t < num_threads; ++t) {
        if (jobs[t].status != 0 && status == 0)
            status = jobs[t].status;
        skipped += jobs[t].skipped;
    }
    if (skipped_out)
        *skipped_out = skipped;
    return status;
}

int orc_paged_attention(double *out, const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, const int32_t *context_lens,
                        int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                        int block_size, double scale, int window, int dtype,
                        int max_blocks_per_seq, int num_blocks, int invalid_policy,
                        const int32_t *pairs, int64_t num_pairs, int num_threads,
                        int64_t *skipped_out)
{
    if (dtype != ORC_F32 && dtype != ORC_F16 && dtype != ORC_BF16)
        return -4;
    return orc_paged_attention_cache(out, q, k_cache, v_cache, block_tables, context_lens,
                                     num_seqs, num_heads, num_kv_heads, head_dim, block_size, scale,
                                     window, dtype, dtype, max_blocks_per_seq, num_blocks,
                                     invalid_policy, pairs, num_pairs, num_threads, skipped_out);
}

/* ------------------------------------------------------------------ */
/* Append: "each generated token's key/value is saved" into its slot
 * (核心要点), with slot = physical * block_size + offset (案例 2).
 * k, v: [num_tokens][num_kv_heads][head_dim]; a slot < 0 is padding and is
 * skipped; a slot beyond the pool is skipped and counted.  Two tokens naming
 * the same slot make the result depend on order, so that input is refused
 * (-2) before anything is written.  Returns the number of out-of-range slots
 * (>= 0) or a negative error.
 */
int64_t orc_append_kv(void *k_cache, void *v_cache, const void *k, const void *v,
                      const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                      int head_dim, int block_size, int num_blocks, int elt_bytes)
{
    const int64_t pool_slots = (int64_t)num_blocks * block_size;
    for (int64_t i = 0; i < num_tokens; ++i)
        for (int64_t j = 0; j < i; ++j)
            if (slot_mapping[i] >= 0 && slot_mapping[i] == slot_mapping[j])
                return -2;
    const size_t row_bytes = (size_t)head_dim * (size_t)elt_bytes;
    int64_t bad = 0;
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= pool_slots) {
            ++bad;
            continue;
        }
        const int64_t phys = slot / block_size;
        const int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t dst_row = (phys * num_kv_heads + h) * block_size + off;
            const int64_t src_row = i * num_kv_heads + h;
            memcpy((char *)k_cache + dst_row * row_bytes, (const char *)k + src_row * row_bytes, row_bytes);
            memcpy((char *)v_cache + dst_row * row_bytes, (const char *)v + src_row * row_bytes, row_bytes);
        }
    }
    return bad;
}

/* Quantise-on-append: token i's K and V rows (in_dtype) are quantised row by
 * row (orc_quantize_row); the codes go to row `offset` of the slot's page and
 * the scale to the page's scale rows (8-bit page layout above).  Slots as
 * orc_append_kv (padding, out-of-range count, duplicates refused). */
int64_t orc_append_kv_quant(void *k_pages, void *v_pages, const void *k, const void *v,
                            const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, int in_dtype, int fmt)
{
    if ((fmt != ORC_I8 && fmt != ORC_E4M3) ||
        (in_dtype != ORC_F32 && in_dtype != ORC_F16 && in_dtype != ORC_BF16))
        return -4;
    const int64_t pool_slots = (int64_t)num_blocks * block_size;
    for (int64_t i = 0; i < num_tokens; ++i)
        for (int64_t j = 0; j < i; ++j)
            if (slot_mapping[i] >= 0 && slot_mapping[i] == slot_mapping[j])
                return -2;
    const int64_t page_bytes = (int64_t)(block_size + orc_scale_rows(block_size, head_dim)) * head_dim;
    int64_t bad = 0;
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= pool_slots) {
            ++bad;
            continue;
        }
        const int64_t phys = slot / block_size;
        const int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t page = phys * num_kv_heads + h;
            const int64_t src_row = i * num_kv_heads + h;
            uint8_t *kp = (uint8_t *)k_pages + page * page_bytes;
            uint8_t *vp = (uint8_t *)v_pages + page * page_bytes;
            float ks, vs;
            orc_quantize_row(k, in_dtype, src_row, head_dim, fmt, kp + off * head_dim, &ks);
            orc_quantize_row(v, in_dtype, src_row, head_dim, fmt, vp + off * head_dim, &vs);
            memcpy(kp + (int64_t)block_size * head_dim + 4 * off, &ks, 4);
            memcpy(vp + (int64_t)block_size * head_dim + 4 * off, &vs, 4);
        }
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Copy-on-write block copy (案例 3: the copy granularity is one block).
 * pairs: int64 [num_pairs][2] = (src, dst).  A pair naming a block outside the
 * pool is skipped and counted.  A destination that repeats, or that is also a
 * source, makes the result order-dependent and is refused (-2).
 */
int64_t orc_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int64_t num_pairs,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        int elt_bytes)
{
    for (int64_t i = 0; i < num_pairs; ++i)
        for (int64_t j = 0; j < num_pairs; ++j) {
            if (i != j && pairs[2 * i + 1] == pairs[2 * j + 1])
                return -2;
            if (pairs[2 * i + 1] == pairs[2 * j])
                return -2;
        }
    const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * elt_bytes;
    int64_t bad = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            ++bad;
            continue;
        }
        memcpy((char *)k_cache + dst * block_bytes, (const char *)k_cache + src * block_bytes, block_bytes);
        memcpy((char *)v_cache + dst * block_bytes, (const char *)v_cache + src * block_bytes, block_bytes);
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Swap: the block copy between two pools (one of them in host memory on the
 * GPU side).  pairs: int64 [num_pairs][2] = (src block of the source pool,
 * dst block of the destination pool).  A pair outside either pool is skipped
 * and counted; a destination named twice is refused (-2).
 */
int64_t orc_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v, const int64_t *pairs,
                        int64_t num_pairs, int src_num_blocks, int dst_num_blocks, int num_kv_heads,
                        int head_dim, int block_size, int elt_bytes)
{
    for (int64_t i = 0; i < num_pairs; ++i)
        for (int64_t j = 0; j < i; ++j)
            if (pairs[2 * i + 1] == pairs[2 * j + 1])
                return -2;
    const size_t block_bytes = (size_t)num_kv_heads * block_size * head_dim * elt_bytes;
    int64_t bad = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
            ++bad;
            continue;
        }
        memcpy((char *)dst_k + dst * block_bytes, (const char *)src_k + src * block_bytes, block_bytes);
        memcpy((char *)dst_v + dst * block_bytes, (const char *)src_v + src * block_bytes, block_bytes);
    }
    return bad;
}
