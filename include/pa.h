/*
 * pa.h — C ABI of the paged KV-cache library (libpa.so, CUDA for sm_103a).
 *
 * Three operations make up the decode-step hot path of PagedAttention:
 *
 *   pa_decode       attention of one new query per sequence over that
 *                   sequence's cached keys/values, read through its block
 *                   table;
 *   pa_append_kv    store each new token's key/value rows into its slot;
 *   pa_copy_blocks  copy whole blocks, the copy-on-write step for blocks that
 *                   several sequences share;
 *   pa_swap_blocks  copy whole blocks between two pools (GPU memory and host
 *                   memory), the swap step of residency changes.
 *
 * Sources (web pages on PagedAttention):
 *   [A] "PagedAttention: From Operating System Virtual Memory to Large
 *       Language Model Memory Systems", section 2 Background — the attention
 *       formula softmax(Q K^T / sqrt(d)) V; section 4 Core Innovation —
 *       logical KV blocks -> block table -> physical GPU blocks.
 *   [B] "PagedAttention — 把 KV cache 当虚拟内存页来管理", 核心要点 (each
 *       generated token's key/value is saved and re-read on later steps),
 *       实践案例 案例 2 (locate: logical block t / block_size through the
 *       table, offset t % block_size; the attention kernel does this one
 *       extra lookup), 案例 3 (reference counts, copy-on-write, one block is
 *       the copy unit), 踩过的坑 (16-token blocks are the default).
 *   [C] "KV Cache与长上下文管理", section "让 Round Robin / Sliding Window 变成
 *       O(1) 操作" — a sliding window by recycling pages and rewriting the
 *       page table, with no K/V movement.
 *   [D] "PagedAttention 的技术溯源与演进脉络" (mjmagnets article), section 2.2
 *       — a long sequence is cut into several attention units; here those are
 *       the context partitions merged by a log-sum-exp reduce.
 *
 * Memory and ownership.  Every pointer argument is DEVICE memory owned by the
 * caller unless stated otherwise; the library allocates nothing, keeps no
 * per-call state and never synchronises: all work is enqueued on `stream`
 * (a cudaStream_t; NULL means the legacy default stream).  The functions are
 * thread-safe.  The library's state: a per-device cache of SM count and
 * kernel occupancy, filled on first use, and a pool of item counters in
 * device memory (module scope, zero when the library loads).  A decode
 * kernel that claims its items from a counter takes a {next item, CTAs done}
 * pair for its launch and its last CTA returns it to zero.  Eager launches
 * take pairs round-robin from 4096, so at most 4096 decode launches may be in
 * flight at once.  A launch captured into a CUDA graph keeps its pair for
 * every replay, so it takes one of another 4096 pairs for good (no eager or
 * other captured launch ever shares it); once those are spent, captured
 * launches schedule their items statically (the same results).  Two
 * instances of one captured graph must not run at the same time (they would
 * share the counter, as they share out and the workspace).
 *
 * Layouts (row-major, densely packed):
 *   q, out           [num_seqs][num_heads][head_dim]
 *   k_cache, v_cache [num_blocks][num_kv_heads][block_size][head_dim]
 *                    (one (block, kv head) tile is contiguous)
 *   block_tables     int32 [num_seqs][max_blocks_per_seq]
 *   context_lens     int32 [num_seqs]
 *   k, v (append)    [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping     int64 [num_tokens], slot = physical_block * block_size + offset
 *   src_dst_pairs    int64 [num_pairs][2]
 * Query head h reads kv head h / (num_heads / num_kv_heads).
 *
 * Errors.  Bad scalar arguments, null pointers, misaligned pointers (q,
 * caches, k, v must be 16-byte aligned) and a too-small workspace are found
 * on the host before anything is launched (PA_ERR_*).  Bad array CONTENTS on
 * the device (a table entry outside [0, num_blocks), a slot or pair outside
 * the pool) are never dereferenced: the token, row or pair is skipped and a
 * bit is OR-ed into *err_word (a device uint32, nullable, sticky: the caller
 * clears and reads it).  No kernel traps or asserts.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef struct CUstream_st *pa_stream_t; /* same type as cudaStream_t */

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARGUMENT = 1, /* null pointer, negative size, misalignment, bad enum */
    PA_ERR_UNSUPPORTED = 2,      /* a shape or dtype the library does not implement */
    PA_ERR_WORKSPACE_TOO_SMALL = 3,
    PA_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    PA_ERR_NO_BLOCKS = 5         /* block manager: the free list is empty */
} pa_status;

typedef enum {
    PA_F32 = 0,
    PA_F16 = 1,
    PA_BF16 = 2,
    PA_I8 = 3,   /* 8-bit cache codes: two's-complement integers (with row scales) */
    PA_E4M3 = 4  /* 8-bit cache codes: OCP FP8 E4M3 (with row scales) */
} pa_dtype;

/* Bits OR-ed into *err_word by the kernels. */
#define PA_DEVERR_BAD_BLOCK 0x1u /* decode: table entry outside [0, num_blocks); its tokens were left out */
#define PA_DEVERR_BAD_SLOT 0x2u  /* append: slot >= num_blocks * block_size; the row was not written */
#define PA_DEVERR_BAD_PAIR 0x4u  /* copy: src or dst outside [0, num_blocks); the pair was skipped */
#define PA_DEVERR_TIMEOUT 0x8u   /* a pipeline wait gave up (about 2 s); the output is not valid */
#define PA_DEVERR_BAD_LEN 0x10u  /* decode: context_lens[s] > max_blocks_per_seq * block_size; clamped to that */
#define PA_DEVERR_BAD_LAUNCH 0x20u /* a kernel refused its launch configuration; the output is not valid */

/*
 * Bytes of scratch pa_decode needs for split-context partials (0 when no
 * sequence can span more than one partition).  The arguments mean the same as
 * in pa_decode; partition_size 0 selects the default.  The workspace holds,
 * per (sequence, query head, partition), the running max, the softmax
 * denominator and the unnormalised output row in fp32.
 */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int block_size,
                                int max_blocks_per_seq, int window, int partition_size);

/*
 * Paged decode attention [A][B][C][D].
 *
 * For each sequence s and query head h, with L = context_lens[s] and the
 * attended tokens t in [max(0, L - window), L) when window > 0, else [0, L):
 *   k_t = k_cache[table[s][t / block_size]][h / G][t % block_size][:] (same for v_t)
 *   x_t = scale * <q[s][h], k_t>
 *   out[s][h] = sum_t exp(x_t - max x) v_t / sum_t exp(x_t - max x)
 * out[s][h] is 0 when no token is attended (L == 0).  Only table entries of
 * attended tokens are read: a sliding window is expressed purely by rewriting
 * table rows (entries of tokens outside the window may hold anything).
 *
 * Arguments (the ones every paged decode takes first, in that order):
 *   out           [num_seqs][num_heads][head_dim] of out_dtype (written)
 *   q             [num_seqs][num_heads][head_dim] of dtype
 *   k_cache, v_cache  pool of dtype, layout above
 *   block_tables, context_lens  int32, layout above
 *   num_heads % num_kv_heads == 0 and num_heads / num_kv_heads in {1, 2, 4, 8}
 *   head_dim in {64, 128}; block_size in {8, 16, 32}
 *   scale         usually 1 / sqrt(head_dim)
 *   window        0 = whole context, > 0 = last `window` tokens
 *   dtype         element type of q, k_cache and v_cache
 *   out_dtype     element type of out (fp32 keeps the full accuracy)
 *   max_blocks_per_seq  row stride of block_tables; every context must fit:
 *                 context_lens[s] <= max_blocks_per_seq * block_size
 *   num_blocks    pool size, for the bounds check of table entries
 *   partition_size  tokens per context partition, a multiple of block_size,
 *                 at most 256 blocks; 0 = default: 1024 tokens for grouped
 *                 heads (2, 4 or 8 per kv head) with fp16 / bf16 K/V and
 *                 head_dim 128 (the tensor-core kernel), else 512 tokens
 *                 (pa_decode_workspace_size with 0 covers both)
 *   workspace, workspace_bytes  scratch of at least pa_decode_workspace_size()
 *                 bytes (may be NULL when that size is 0)
 *   err_word      device uint32 or NULL
 * num_seqs == 0 returns PA_OK without launching.
 * The same inputs give the same bits on every call: each (sequence, kv head,
 * partition) is computed in a fixed order whichever CTA takes it, and the
 * partitions merge in a fixed order.  (A sequence decoded in batches of a
 * different size may differ in the last bits: the merge picks its layout by
 * the number of rows.)
 */
PA_API pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *context_lens,
                    int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                    int block_size, float scale, int window,
                    pa_dtype dtype, pa_dtype out_dtype, int max_blocks_per_seq,
                    int num_blocks, int partition_size, void *workspace,
                    size_t workspace_bytes, uint32_t *err_word, pa_stream_t stream);

/*
 * Decode attention for groups of sequences that share a prompt prefix [B
 * 核心要点 and 案例 3: parallel samples of one prompt share its blocks].  Same
 * result as pa_decode (window 0) for every sequence; the shared blocks are
 * read once per group instead of once per sequence.
 *   Sequences come in consecutive groups of group_size (num_seqs a multiple
 *   of it).  Group g's members share their first shared_lens[g] tokens: their
 *   block tables agree on the first shared_lens[g] / block_size entries (as a
 *   fork produces).  The shared blocks are read through the first member's
 *   table row.  shared_lens is a device int32 [num_seqs / group_size]; each
 *   value is used rounded down to whole blocks and to at most every member's
 *   context (PA_DEVERR_BAD_LEN flags a change).
 *   Supported: fp16 / bf16 K/V, head_dim 128, group_size * (num_heads /
 *   num_kv_heads) in {2, 4, 8} (the grouped queries of one kv head go
 *   through the tensor-core kernel together).
 *   workspace: at least pa_decode_shared_prefix_workspace_size() bytes,
 *   16-byte aligned (regrouped queries, lengths, two sets of partials).
 * Other arguments as pa_decode.
 */
PA_API pa_status pa_decode_shared_prefix(void *out, const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, const int32_t *context_lens,
                                         const int32_t *shared_lens, int group_size, int num_seqs,
                                         int num_heads, int num_kv_heads, int head_dim, int block_size,
                                         float scale, pa_dtype dtype, pa_dtype out_dtype,
                                         int max_blocks_per_seq, int num_blocks, int partition_size,
                                         void *workspace, size_t workspace_bytes, uint32_t *err_word,
                                         pa_stream_t stream);

/* Bytes of workspace pa_decode_shared_prefix needs (0 for bad arguments). */
PA_API size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int num_heads, int head_dim,
                                                     int block_size, int max_blocks_per_seq,
                                                     int partition_size, int group_size, pa_dtype dtype);

/*
 * pa_decode without any allocation.  No page describes this call: it exists
 * for callers that cannot allocate device memory (a plugin whose host
 * framework owns all device allocations, a runtime with a fixed memory
 * budget, a path that must not pay for cudaMalloc).  Arguments and results
 * are those of pa_decode without workspace / workspace_bytes: the scratch for
 * partition partials is one array built into the library,
 * pa_decode_noalloc_max_scratch() bytes (32 MiB), which every GPU that loads
 * the library holds until the process exits.
 *  - A shape whose pa_decode_workspace_size() exceeds that size is rejected
 *    with PA_ERR_WORKSPACE_TOO_SMALL before anything is launched, once every
 *    other argument has passed pa_decode's checks (a bad argument is
 *    reported as itself first).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make
 *    that first call before any stream capture.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents (nothing in it needs to start at zero).  Calls that overlap on
 *    the GPU race on it: order them on one stream.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 */
PA_API pa_status pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int window,
                                   pa_dtype dtype, pa_dtype out_dtype, int max_blocks_per_seq,
                                   int num_blocks, int partition_size, uint32_t *err_word,
                                   pa_stream_t stream);

/* Size in bytes of the scratch array pa_decode_noalloc uses. */
PA_API size_t pa_decode_noalloc_max_scratch(void);

/*
 * Decode attention over CONTIGUOUS (non-paged) caches, the baseline for the
 * cost of the block table [B 踩过的坑: the lookup makes the attention kernel
 * 20-26% slower].  The same attention as pa_decode (window, partitions,
 * output dtypes, error word), with no block table: sequence s's token t of
 * kv head h is row t of
 *   k_cache, v_cache [num_seqs][num_kv_heads][max_context_len][head_dim].
 * The kernels are pa_decode's (one query head per kv head: the MHA kernel;
 * 2, 4 or 8 with fp16 / bf16 K/V and head_dim 128: the tensor-core kernel,
 * which moves each 128-token tile of a kv head with one copy); the cache is
 * cut into 16-token blocks, so max_context_len must be a positive multiple of
 * 16 and the workspace is pa_decode_workspace_size(num_seqs, num_heads,
 * head_dim, 16, max_context_len / 16, window, partition_size) bytes.  Other
 * shapes return PA_ERR_UNSUPPORTED.  context_lens[s] > max_context_len is
 * clamped and flagged (PA_DEVERR_BAD_LEN).
 */
PA_API pa_status pa_decode_contiguous(void *out, const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                      int head_dim, int max_context_len, float scale, int window, pa_dtype dtype,
                                      pa_dtype out_dtype, int partition_size, void *workspace,
                                      size_t workspace_bytes, uint32_t *err_word, pa_stream_t stream);

/*
 * Append [B 核心要点, 案例 2]: for every token i with slot = slot_mapping[i] >= 0
 *   k_cache[slot / block_size][h][slot % block_size][:] = k[i][h][:]   (all h)
 *   v_cache[...] = v[i][h][:]
 * A bit-exact copy (k, v and the caches share `dtype`).  A negative slot is
 * padding and is skipped; a slot >= num_blocks * block_size is skipped and
 * flagged.  Two tokens naming one slot leave that slot holding one of them
 * (unspecified which): callers must not do this.
 * num_tokens == 0 returns PA_OK without launching.
 */
PA_API pa_status pa_append_kv(const void *k, const void *v, const int64_t *slot_mapping,
                       void *k_cache, void *v_cache, int num_tokens, int num_kv_heads,
                       int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                       uint32_t *err_word, pa_stream_t stream);

/*
 * Copy-on-write block copy [B 案例 3]: for each pair (src, dst) copy block src
 * onto block dst in both caches (all kv heads, all rows).  A pair naming a
 * block outside the pool is skipped and flagged.  A destination that repeats
 * or that is also a source makes the result order-dependent: callers must not
 * do this.  num_pairs == 0 returns PA_OK without launching.
 */
PA_API pa_status pa_copy_blocks(const int64_t *src_dst_pairs, int num_pairs, void *k_cache,
                         void *v_cache, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, pa_dtype dtype, uint32_t *err_word,
                         pa_stream_t stream);

/*
 * Block swap between two pools [B 踩过的坑: swap (or recompute) is the fallback
 * when GPU memory runs short; "PagedAttention的终极用途": pages move between GPU
 * and CPU memory].  For each pair (src, dst) copy block src of the source pool
 * onto block dst of the destination pool, K and V, all kv heads: a bit-exact
 * copy.  Either pool may be device memory or host memory the GPU can address
 * (pinned, mapped host allocations; on GB300 they are reached over the
 * NVLink-C2C host link).  The pairs array must be readable by the GPU too.
 * Both pools share the cache layout, dtype, num_kv_heads, head_dim and
 * block_size.  A pair outside either pool is skipped and flagged
 * (PA_DEVERR_BAD_PAIR).  The pools must not overlap; a destination named
 * twice is order-dependent: callers must not do this.  num_pairs == 0 returns
 * PA_OK without launching.
 */
PA_API pa_status pa_swap_blocks(const int64_t *src_dst_pairs, int num_pairs, const void *src_k,
                                const void *src_v, void *dst_k, void *dst_v, int src_num_blocks,
                                int dst_num_blocks, int num_kv_heads, int head_dim, int block_size,
                                pa_dtype dtype, uint32_t *err_word, pa_stream_t stream);

/*
 * 8-bit KV cache ["KV Cache与长上下文管理": KV-cache quantisation FP16 -> INT8
 * halves the cache; the mjmagnets article, section 4.1: INT8 pages].  The
 * pages fix no scale granularity; this library keeps one fp32 scale per
 * cached (token, kv head) row, so an append quantises only its own rows:
 *   amax = max_j |x_j|,  scale = amax / Q  (one fp32 division; Q = 127 for
 *   PA_I8, 448 for PA_E4M3),
 *   code_j = PA_I8:   round-half-even(x_j / scale) clamped to [-127, 127]
 *            PA_E4M3: x_j / scale (fp32) rounded to the nearest E4M3 value,
 *                     ties to even, saturating at +-448,
 * a row of zeros storing scale 0 and zero codes.  The cached value of an
 * element is code * scale.
 * Pools are pages: k_cache / v_cache are [num_blocks][num_kv_heads][page]
 * with page = pa_quant_page_bytes(head_dim, block_size) bytes: the block's
 * block_size code rows of head_dim bytes (one byte per element), then
 * ceil(4 * block_size / head_dim) rows whose first 4 * block_size bytes are
 * the rows' fp32 scales (little-endian, in row order; the rest is padding).
 * A page moves with one contiguous copy, its scales included.
 */

/* Bytes of one (block, kv head) page of an 8-bit pool (0 for bad arguments). */
PA_API size_t pa_quant_page_bytes(int head_dim, int block_size);

/*
 * Quantise-on-append: token i's K and V rows (dtype PA_F32 / PA_F16 /
 * PA_BF16, [num_tokens][num_kv_heads][head_dim]) are quantised row by row as
 * above; the codes go to row slot % block_size of the slot's page, the scale
 * to the page's scale rows (padding and out-of-range slots as pa_append_kv).
 * cache_dtype is PA_I8 or PA_E4M3.
 */
PA_API pa_status pa_append_kv_quant(const void *k, const void *v, const int64_t *slot_mapping, void *k_cache,
                                    void *v_cache, int num_tokens, int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, pa_dtype dtype, pa_dtype cache_dtype, uint32_t *err_word,
                                    pa_stream_t stream);

/*
 * pa_decode over an 8-bit cache: the same attention with every cached
 * element read as code * scale of its row.  q (dtype PA_F32 / PA_F16 /
 * PA_BF16) and out as pa_decode; cache_dtype PA_I8 or PA_E4M3; the workspace
 * is pa_decode_workspace_size() bytes, as for pa_decode.  partition_size 0
 * selects 1024 tokens for E4M3 pages with fp16 / bf16 queries in groups of 2
 * or 4, head_dim 128, block size 16 or 32 and a multiple of 4 kv heads (the
 * tensor-core kernel), else 512 tokens.
 */
PA_API pa_status pa_decode_quant(void *out, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                                 int num_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                                 int window, pa_dtype dtype, pa_dtype cache_dtype, pa_dtype out_dtype,
                                 int max_blocks_per_seq, int num_blocks, int partition_size, void *workspace,
                                 size_t workspace_bytes, uint32_t *err_word, pa_stream_t stream);

/* pa_copy_blocks for 8-bit pools: whole pages (codes and scales). */
PA_API pa_status pa_copy_blocks_quant(const int64_t *src_dst_pairs, int num_pairs, void *k_cache, void *v_cache,
                                      int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                      uint32_t *err_word, pa_stream_t stream);

/* pa_swap_blocks for 8-bit pools: whole pages (either side may be
 * GPU-addressable host memory, as pa_swap_blocks). */
PA_API pa_status pa_swap_blocks_quant(const int64_t *src_dst_pairs, int num_pairs, const void *src_k,
                                      const void *src_v, void *dst_k, void *dst_v, int src_num_blocks,
                                      int dst_num_blocks, int num_kv_heads, int head_dim, int block_size,
                                      uint32_t *err_word, pa_stream_t stream);

/* Static text for a status code. */
PA_API const char *pa_status_string(pa_status status);

/* Detail of the last PA_ERR_* returned on the calling thread ("" if none). */
PA_API const char *pa_last_error_detail(void);

/* Library version, (major << 16) | (minor << 8) | patch. */
PA_API int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
