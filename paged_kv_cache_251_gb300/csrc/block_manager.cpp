// Host-side KV block manager: free list, reference counts, copy-on-write and
// sliding-window rings.  Interface and sources: include/pa_block_manager.h.
#include <cstdint>
#include <deque>
#include <new>
#include <vector>

#include "pa_block_manager.h"

struct pa_bm {
    struct Seq {
        bool live = false;
        long long length = 0;
        int ring = 0;                   // ring size (0: ordinary sequence)
        std::vector<int32_t> table;     // logical block -> physical block (-1: none / recycled)
        std::vector<int32_t> ring_ids;  // physical blocks of the ring, in ring order
    };
    int num_blocks = 0, block_size = 0, max_seqs = 0, max_blocks = 0;
    std::vector<int32_t> ref;
    std::deque<int32_t> free_list;
    std::vector<Seq> seqs;

    bool take(int32_t *b) {
        if (free_list.empty())
            return false;
        *b = free_list.front();
        free_list.pop_front();
        ref[*b] = 1;
        return true;
    }
    void drop(int32_t b) {
        if (b < 0)
            return;
        if (--ref[b] == 0)
            free_list.push_back(b);
    }
    bool valid(int s) const { return s >= 0 && s < max_seqs; }
};

extern "C" {

pa_bm *pa_bm_create(int num_blocks, int block_size, int max_seqs, int max_blocks_per_seq,
                    const int32_t *free_order) {
    if (num_blocks <= 0 || block_size <= 0 || max_seqs <= 0 || max_blocks_per_seq <= 0)
        return nullptr;
    pa_bm *bm = new (std::nothrow) pa_bm;
    if (!bm)
        return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->max_seqs = max_seqs;
    bm->max_blocks = max_blocks_per_seq;
    bm->ref.assign(num_blocks, 0);
    bm->seqs.resize(max_seqs);
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
        const int32_t b = free_order ? free_order[i] : i;
        if (b < 0 || b >= num_blocks || seen[b]) {
            delete bm;
            return nullptr;
        }
        seen[b] = 1;
        bm->free_list.push_back(b);
    }
    return bm;
}

void pa_bm_destroy(pa_bm *bm) { delete bm; }

pa_status pa_bm_add_sequence(pa_bm *bm, int seq, int ring_blocks) {
    if (!bm || !bm->valid(seq) || bm->seqs[seq].live || ring_blocks < 0)
        return PA_ERR_INVALID_ARGUMENT;
    pa_bm::Seq &s = bm->seqs[seq];
    s = pa_bm::Seq();
    s.live = true;
    s.ring = ring_blocks;
    return PA_OK;
}

pa_status pa_bm_fork(pa_bm *bm, int parent, int child) {
    if (!bm || !bm->valid(parent) || !bm->valid(child) || parent == child || !bm->seqs[parent].live ||
        bm->seqs[child].live || bm->seqs[parent].ring)
        return PA_ERR_INVALID_ARGUMENT;
    const pa_bm::Seq &p = bm->seqs[parent];
    pa_bm::Seq &c = bm->seqs[child];
    c = p;
    for (int32_t b : c.table)
        if (b >= 0)
            ++bm->ref[b];
    return PA_OK;
}

pa_status pa_bm_free_sequence(pa_bm *bm, int seq) {
    if (!bm || !bm->valid(seq) || !bm->seqs[seq].live)
        return PA_ERR_INVALID_ARGUMENT;
    pa_bm::Seq &s = bm->seqs[seq];
    if (s.ring) {
        for (int32_t b : s.ring_ids)
            bm->drop(b);
    } else {
        for (int32_t b : s.table)
            bm->drop(b);
    }
    s = pa_bm::Seq();
    return PA_OK;
}

pa_status pa_bm_append(pa_bm *bm, const int32_t *seqs, int n, int64_t *slots, int64_t *pairs, int pairs_cap,
                       int *num_pairs, int *placed) {
    int np = 0, done = 0;
    pa_status st = PA_OK;
    if (!bm || n < 0 || (n > 0 && !seqs) || pairs_cap < 0 || (pairs_cap > 0 && !pairs))
        st = PA_ERR_INVALID_ARGUMENT;
    for (; st == PA_OK && done < n; ++done) {
        const int sid = seqs[done];
        if (!bm->valid(sid) || !bm->seqs[sid].live) {
            st = PA_ERR_INVALID_ARGUMENT;
            break;
        }
        pa_bm::Seq &s = bm->seqs[sid];
        const long long pos = s.length;
        const long long lb = pos / bm->block_size;
        const int off = static_cast<int>(pos % bm->block_size);
        if (lb >= bm->max_blocks) {
            st = PA_ERR_INVALID_ARGUMENT;  // the table row is full
            break;
        }
        if (s.ring) {
            if (off == 0) {  // entering a new logical block: recycle through the ring
                const int r = static_cast<int>(lb % s.ring);
                if (static_cast<int>(s.ring_ids.size()) <= r) {
                    int32_t b;
                    if (!bm->take(&b)) {
                        st = PA_ERR_NO_BLOCKS;
                        break;
                    }
                    s.ring_ids.push_back(b);
                }
                if (static_cast<long long>(s.table.size()) <= lb)
                    s.table.resize(lb + 1, -1);
                if (lb >= s.ring)
                    s.table[lb - s.ring] = -1;  // its page now holds the new block
                s.table[lb] = s.ring_ids[r];
            }
        } else {
            if (static_cast<long long>(s.table.size()) == lb) {  // a block on demand
                int32_t b;
                if (!bm->take(&b)) {
                    st = PA_ERR_NO_BLOCKS;
                    break;
                }
                s.table.push_back(b);
            }
            const int32_t cur = s.table[lb];
            if (bm->ref[cur] > 1) {  // shared: copy-on-write
                if (np >= pairs_cap) {
                    st = PA_ERR_INVALID_ARGUMENT;  // no room to report the copy
                    break;
                }
                int32_t fresh;
                if (!bm->take(&fresh)) {
                    st = PA_ERR_NO_BLOCKS;
                    break;
                }
                --bm->ref[cur];
                pairs[2 * np] = cur;
                pairs[2 * np + 1] = fresh;
                ++np;
                s.table[lb] = fresh;
            }
        }
        if (slots)
            slots[done] = static_cast<int64_t>(s.table[lb]) * bm->block_size + off;
        s.length = pos + 1;
    }
    if (num_pairs)
        *num_pairs = np;
    if (placed)
        *placed = done;
    return st;
}

long long pa_bm_length(const pa_bm *bm, int seq) {
    if (!bm || !bm->valid(seq) || !bm->seqs[seq].live)
        return -1;
    return bm->seqs[seq].length;
}

pa_status pa_bm_tables(const pa_bm *bm, int32_t *tables, int32_t *lens) {
    if (!bm)
        return PA_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < bm->max_seqs; ++i) {
        const pa_bm::Seq &s = bm->seqs[i];
        if (tables) {
            int32_t *row = tables + static_cast<long long>(i) * bm->max_blocks;
            for (int j = 0; j < bm->max_blocks; ++j)
                row[j] = (s.live && j < static_cast<int>(s.table.size())) ? s.table[j] : -1;
        }
        if (lens)
            lens[i] = s.live ? static_cast<int32_t>(s.length) : 0;
    }
    return PA_OK;
}

int pa_bm_refcount(const pa_bm *bm, int block) {
    if (!bm || block < 0 || block >= bm->num_blocks)
        return -1;
    return bm->ref[block];
}

int pa_bm_num_free(const pa_bm *bm) { return bm ? static_cast<int>(bm->free_list.size()) : -1; }

}  // extern "C"
