/*
 * pa_block_manager.h — host-side KV block manager of libpa (C ABI, CPU only).
 *
 * It owns no K/V bytes: it decides which physical block and offset each new
 * token goes to, and it produces the three inputs of the device calls —
 * block tables (pa_decode), slot mappings (pa_append_kv) and copy-on-write
 * (src, dst) pairs (pa_copy_blocks).
 *
 * Sources (web pages on PagedAttention):
 *   [B] "PagedAttention — 把 KV cache 当虚拟内存页来管理": 核心要点 (a sequence
 *       sees contiguous logical blocks while physical blocks are scattered;
 *       blocks are taken on demand), 实践案例 案例 2 (slot of token t =
 *       table[t / block_size] * block_size + t % block_size), 案例 3 (blocks
 *       carry reference counts; a write into a block shared by more than one
 *       sequence first drops one reference, takes a fresh block, copies the
 *       old block into it and writes there; the sole owner writes in place;
 *       one block is the copy unit).
 *   [C] "KV Cache与长上下文管理", section "让 Round Robin / Sliding Window 变成
 *       O(1) 操作": a sliding window recycles the oldest page and rewrites only
 *       the page table; no K/V data moves.  Here a window sequence owns a ring
 *       of R physical blocks; logical block lb lives in ring[lb % R], and
 *       entering a new logical block rewrites two table entries (the new one,
 *       and the recycled one, which becomes -1).  For a token-exact window of
 *       W tokens, R = ceil(W / block_size) + 1 keeps every attended token
 *       resident.
 *
 * Thread safety: a manager is not internally locked; use one per thread or
 * lock around calls.  All arrays are host memory owned by the caller.
 * Errors are returned as pa_status (pa.h); PA_ERR_NO_BLOCKS when the pool is
 * exhausted.
 */
#ifndef PA_BLOCK_MANAGER_H
#define PA_BLOCK_MANAGER_H

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_bm pa_bm;

/*
 * A manager for a pool of num_blocks physical blocks of block_size tokens,
 * up to max_seqs sequences (ids 0 .. max_seqs-1) whose tables hold up to
 * max_blocks_per_seq entries.  free_order (nullable, num_blocks distinct ids)
 * is the order in which free blocks are handed out; NULL means 0, 1, 2, ...
 * Returns NULL on bad arguments.
 */
PA_API pa_bm *pa_bm_create(int num_blocks, int block_size, int max_seqs, int max_blocks_per_seq,
                           const int32_t *free_order);
PA_API void pa_bm_destroy(pa_bm *bm);

/* Start an empty sequence.  ring_blocks 0: an ordinary sequence; > 0: a
 * sliding-window sequence over a ring of that many physical blocks. */
PA_API pa_status pa_bm_add_sequence(pa_bm *bm, int seq, int ring_blocks);

/* child shares every block of parent (each block's count goes up by one) and
 * takes parent's length.  Not available for window sequences. */
PA_API pa_status pa_bm_fork(pa_bm *bm, int parent, int child);

/* Drop a sequence; blocks whose count reaches zero return to the free list. */
PA_API pa_status pa_bm_free_sequence(pa_bm *bm, int seq);

/*
 * Place n new tokens: token i goes to the end of sequence seqs[i] (tokens of
 * one sequence in the order given).  slots[i] (nullable) receives its slot.
 * Each copy-on-write needed is recorded as (src, dst) in pairs[2 * k] (at
 * most pairs_cap pairs; nullable when pairs_cap is 0 and none is needed).
 * *num_pairs receives the count, *placed the number of tokens placed (n on
 * success).  On PA_ERR_NO_BLOCKS or a full table the tokens before the
 * failing one stay placed.
 */
PA_API pa_status pa_bm_append(pa_bm *bm, const int32_t *seqs, int n, int64_t *slots, int64_t *pairs,
                              int pairs_cap, int *num_pairs, int *placed);

/* Tokens held by a sequence (-1 if it does not exist). */
PA_API long long pa_bm_length(const pa_bm *bm, int seq);

/* Export block tables int32 [max_seqs][max_blocks_per_seq] (entries not in
 * use, and recycled window entries, are -1) and lengths int32 [max_seqs]
 * (0 for absent sequences).  Either pointer may be NULL. */
PA_API pa_status pa_bm_tables(const pa_bm *bm, int32_t *tables, int32_t *lens);

/* Reference count of a physical block (0 = free), -1 if out of range. */
PA_API int pa_bm_refcount(const pa_bm *bm, int block);

/* Number of blocks on the free list. */
PA_API int pa_bm_num_free(const pa_bm *bm);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H */
