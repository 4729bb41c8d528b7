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
 *    page table; the attended set is the most recent tokens.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

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
            dot += orc_load(a->q, a->dtype, q_base + j) * orc_load(a->k_cache, a->dtype, row[i] + j);
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
            out_row[j] += w * orc_load(a->v_cache, a->dtype, row[i] + j);
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
int orc_paged_attention(double *out, const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, const int32_t *context_lens,
                        int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                        int block_size, double scale, int window, int dtype,
                        int max_blocks_per_seq, int num_blocks, int invalid_policy,
                        const int32_t *pairs, int64_t num_pairs, int num_threads,
                        int64_t *skipped_out)
{
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || (dtype != ORC_F32 && dtype != ORC_F16 && dtype != ORC_BF16))
        return -4;
    orc_args a = {q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                  num_kv_heads, head_dim, block_size, scale, window, dtype,
                  max_blocks_per_seq, num_blocks, invalid_policy};
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
