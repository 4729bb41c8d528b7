// Decode attention for groups of sequences that share a prompt prefix
// ("PagedAttention — 把 KV cache 当虚拟内存页来管理", 核心要点 and 案例 3:
// parallel samples of one prompt point their block tables at the same prompt
// blocks).  The result is exactly pa_decode's; what changes is how often the
// shared blocks are read: once per group instead of once per sequence.
//
//   prep     per group, the usable shared length (whole blocks, at most every
//            member's context); per sequence, where its own tokens start; the
//            group members' queries regrouped so that, for one kv head, the
//            group_size x G query heads are consecutive rows;
//   prefix   the grouped-query decode kernel over the shared blocks, one
//            "sequence" per group whose query heads are all members' heads:
//            each shared K/V tile is read once and multiplied against
//            group_size x G queries on the tensor cores; partials only;
//   suffix   the usual decode kernel over each sequence's tokens after the
//            shared prefix; partials only;
//   combine  per (sequence, head), the log-sum-exp merge of the prefix and
//            suffix partials into the output.
#include <cuda_runtime.h>

#include <climits>
#include <string>

#include "pa.h"
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kDefaultPartitionTokens = 512;
constexpr int kGqaDefaultPartitionTokens = 1024;  // the prefix pass (tensor-core kernel)

__global__ void __launch_bounds__(256)
    prefix_prep_kernel(const int32_t *__restrict__ context_lens, const int32_t *__restrict__ shared_lens,
                       int32_t *shared_eff, int32_t *start_tok, const uint4 *__restrict__ q, uint4 *qv,
                       int num_groups, int group_size, int num_heads, int num_kv_heads, int chunks_per_row,
                       int block_size, int max_len, uint32_t *err) {
    pdl_launch_dependents();
    pdl_wait();
    const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long g = tid; g < num_groups; g += stride) {
        const int want = shared_lens[g];
        int eff = want < 0 ? 0 : want / block_size * block_size;
        for (int j = 0; j < group_size; ++j) {
            int L = context_lens[g * group_size + j];
            L = L < 0 ? 0 : (L > max_len ? max_len : L);
            const int whole = L / block_size * block_size;
            if (whole < eff)
                eff = whole;
        }
        if (eff != want && err)
            atomicOr(err, PA_DEVERR_BAD_LEN);
        shared_eff[g] = eff;
        for (int j = 0; j < group_size; ++j)
            start_tok[g * group_size + j] = eff;
    }
    // regroup the queries: row (s, h) -> (group, kv head, member, head in group)
    const int G = num_heads / num_kv_heads;
    const int Gp = group_size * G;
    const long long total = static_cast<long long>(num_groups) * group_size * num_heads * chunks_per_row;
    for (long long idx = tid; idx < total; idx += stride) {
        const long long row = idx / chunks_per_row;
        const int c = static_cast<int>(idx - row * chunks_per_row);
        const int h = static_cast<int>(row % num_heads);
        const long long s = row / num_heads;
        const long long g = s / group_size;
        const int j = static_cast<int>(s - g * group_size);
        const int kvh = h / G, gg = h - kvh * G;
        const long long dst = (g * num_kv_heads + kvh) * Gp + j * G + gg;
        qv[dst * chunks_per_row + c] = q[idx];
    }
}

// One warp per (sequence, head), kReduceRows rows per CTA: merge the prefix
// pass's partials of its group row with the suffix pass's partials of its own
// row.  The partitions are taken kBatch at a time, their (m, l) pairs and
// head_dim slices all loaded before any is used, and folded into a running
// max, denominator and numerator.
template <int D>
__global__ void __launch_bounds__(kReduceThreads)
    prefix_combine_kernel(const DecodeParams pre, const DecodeParams suf, const int32_t *__restrict__ shared_eff,
                          int group_size) {
    constexpr int kPer = D / 32;  // head_dim slice per lane (4 or 2)
    constexpr int kBatch = 8;
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long rowi = static_cast<long long>(blockIdx.x) * kReduceRows + (threadIdx.x >> 5);  // s * H + h
    if (rowi >= static_cast<long long>(suf.num_seqs) * suf.num_heads)
        return;
    const int H = suf.num_heads, G = suf.num_heads / suf.num_kv_heads;
    const long long s = rowi / H;
    const int h = static_cast<int>(rowi - s * H);
    const long long g = s / group_size;
    const int j = static_cast<int>(s - g * group_size);
    const int kvh = h / G, gg = h - kvh * G;
    const long long rowp = (g * suf.num_kv_heads + kvh) * (group_size * G) + j * G + gg;
    const int eff = ld_nc_i32(shared_eff + g);
    const int len = ld_nc_i32(suf.context_lens + s);
    const int np_pre = seq_span(eff, pre.max_len, 0, pre.block_size, pre.bpp).nparts;
    const int np_suf = seq_span(len, suf.max_len, 0, suf.block_size, suf.bpp, eff).nparts;
    const int np = np_pre + np_suf;
    const float2 *ml_pre = reinterpret_cast<const float2 *>(pre.part_ml + rowp * pre.max_parts * 2);
    const float2 *ml_suf = reinterpret_cast<const float2 *>(suf.part_ml + rowi * suf.max_parts * 2);
    const float *acc_pre = pre.part_acc + rowp * pre.max_parts * D + lane * kPer;
    const float *acc_suf = suf.part_acc + rowi * suf.max_parts * D + lane * kPer;

    float mw = -INFINITY, dw = 0.f, nw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        nw[i] = 0.f;
    for (int q0 = 0; q0 < np; q0 += kBatch) {
        float2 m[kBatch];
        float v[kBatch][kPer];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int q = q0 + b;
            m[b] = make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                v[b][i] = 0.f;
            if (q < np) {
                const bool in_pre = q < np_pre;
                m[b] = in_pre ? ml_pre[q] : ml_suf[q - np_pre];
                const float *a = in_pre ? acc_pre + static_cast<long long>(q) * D
                                        : acc_suf + static_cast<long long>(q - np_pre) * D;
                if constexpr (kPer == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(a);
                    v[b][0] = x.x, v[b][1] = x.y, v[b][2] = x.z, v[b][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(a);
                    v[b][0] = x.x, v[b][1] = x.y;
                }
            }
        }
        float bm = -INFINITY;
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
            bm = fmaxf(bm, m[b].x);
        const float mn = fmaxf(mw, bm);
        if (mn == -INFINITY)
            continue;
        const float al = mw == -INFINITY ? 0.f : exp2f(mw - mn);
        dw *= al;
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            nw[i] *= al;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            if (m[b].x != -INFINITY) {
                const float sc = exp2f(m[b].x - mn);
                dw = fmaf(m[b].y, sc, dw);
#pragma unroll
                for (int i = 0; i < kPer; ++i)
                    nw[i] = fmaf(v[b][i], sc, nw[i]);
            }
        }
        mw = mn;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        store_out(suf.out, suf.out_dtype, rowi * D + lane * kPer + i, dw > 0.f ? nw[i] / dw : 0.f);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct PrefixPlan {
    int bpp = 0, max_parts = 0;
    size_t q_off = 0, eff_off = 0, start_off = 0, pre_off = 0, suf_off = 0, total = 0;
};

bool plan_prefix(int num_seqs, int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                 int partition_size, int group_size, int elt, PrefixPlan *pl) {
    if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
        group_size <= 0 || num_seqs % group_size != 0)
        return false;
    const int P = partition_size == 0 ? kDefaultPartitionTokens : partition_size;
    if (P <= 0 || P % block_size != 0 || P / block_size > kMaxBpp)
        return false;
    pl->bpp = P / block_size;
    pl->max_parts = (max_blocks_per_seq + pl->bpp - 1) / pl->bpp;
    const size_t rows = static_cast<size_t>(num_seqs) * num_heads;
    const size_t part_bytes = rows * pl->max_parts * (head_dim + 2) * sizeof(float);
    pl->q_off = 0;
    pl->eff_off = align256(rows * head_dim * elt);
    pl->start_off = align256(pl->eff_off + sizeof(int32_t) * (num_seqs / group_size));
    pl->pre_off = align256(pl->start_off + sizeof(int32_t) * num_seqs);
    pl->suf_off = align256(pl->pre_off + part_bytes);
    pl->total = align256(pl->suf_off + part_bytes);
    return true;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int num_heads, int head_dim, int block_size,
                                                         int max_blocks_per_seq, int partition_size, int group_size,
                                                         pa_dtype dtype) {
    PrefixPlan pl;
    if (!plan_prefix(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq, partition_size, group_size,
                     dtype == PA_F32 ? 4 : 2, &pl))
        return 0;
    return pl.total;
}

extern "C" pa_status pa_decode_shared_prefix(void *out, const void *q, const void *k_cache, const void *v_cache,
                                             const int32_t *block_tables, const int32_t *context_lens,
                                             const int32_t *shared_lens, int group_size, int num_seqs, int num_heads,
                                             int num_kv_heads, int head_dim, int block_size, float scale,
                                             pa_dtype dtype, pa_dtype out_dtype, int max_blocks_per_seq,
                                             int num_blocks, int partition_size, void *workspace,
                                             size_t workspace_bytes, uint32_t *err_word, pa_stream_t stream) {
    auto bad = [](pa_status st, const char *why) {
        set_last_error_detail(why);
        return st;
    };
    set_last_error_detail("");
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
        max_blocks_per_seq <= 0 || num_blocks <= 0 || group_size <= 0)
        return bad(PA_ERR_INVALID_ARGUMENT, "sizes out of range, or num_heads not a multiple of num_kv_heads");
    if (num_seqs % group_size != 0)
        return bad(PA_ERR_INVALID_ARGUMENT, "num_seqs must be a multiple of group_size");
    if (num_seqs == 0)
        return PA_OK;
    const int G = num_heads / num_kv_heads;
    const int Gp = group_size * G;
    if (head_dim != 128 || (dtype != PA_F16 && dtype != PA_BF16))
        return bad(PA_ERR_UNSUPPORTED, "the shared-prefix decode takes fp16 / bf16 K/V with head_dim 128");
    if (Gp != 2 && Gp != 4 && Gp != 8)
        return bad(PA_ERR_UNSUPPORTED, "group_size * (num_heads / num_kv_heads) must be 2, 4 or 8");
    if (block_size != 8 && block_size != 16 && block_size != 32)
        return bad(PA_ERR_UNSUPPORTED, "block_size must be 8, 16 or 32");
    if (out_dtype != PA_F32 && out_dtype != PA_F16 && out_dtype != PA_BF16)
        return bad(PA_ERR_INVALID_ARGUMENT, "unknown dtype");
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !shared_lens)
        return bad(PA_ERR_INVALID_ARGUMENT, "null pointer");
    auto a16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(workspace))
        return bad(PA_ERR_INVALID_ARGUMENT, "q, the caches and the workspace must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(out) & ((out_dtype == PA_F32 ? 4 : 2) - 1)) != 0)
        return bad(PA_ERR_INVALID_ARGUMENT, "out is not aligned to its element size");
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
        return bad(PA_ERR_INVALID_ARGUMENT, "scale must be finite");
    PrefixPlan pl;
    if (!plan_prefix(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq, partition_size, group_size, 2,
                     &pl))
        return bad(PA_ERR_INVALID_ARGUMENT, "partition_size must be a positive multiple of block_size, at most 256 blocks");
    if (!workspace || workspace_bytes < pl.total)
        return bad(PA_ERR_WORKSPACE_TOO_SMALL, "workspace smaller than pa_decode_shared_prefix_workspace_size()");
    if (static_cast<long long>(max_blocks_per_seq) * group_size > INT_MAX)
        return bad(PA_ERR_UNSUPPORTED, "table rows too long for the grouped view");

    char *ws = static_cast<char *>(workspace);
    void *qv = ws + pl.q_off;
    int32_t *shared_eff = reinterpret_cast<int32_t *>(ws + pl.eff_off);
    int32_t *start_tok = reinterpret_cast<int32_t *>(ws + pl.start_off);
    const int num_groups = num_seqs / group_size;
    const int max_len = static_cast<int>(
        static_cast<long long>(max_blocks_per_seq) * block_size > INT_MAX ? INT_MAX
                                                                           : max_blocks_per_seq * block_size);
    const size_t acc_floats = static_cast<size_t>(num_seqs) * num_heads * pl.max_parts * head_dim;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

    // 1) shared lengths, start tokens, regrouped queries
    const int cpr = head_dim * 2 / 16;
    long long work = static_cast<long long>(num_seqs) * num_heads * cpr;
    long long blocks = (work + 255) / 256;
    if (blocks > 4096)
        blocks = 4096;
    if (blocks < 1)
        blocks = 1;
    const uint4 *qs = static_cast<const uint4 *>(q);
    uint4 *qvs = static_cast<uint4 *>(qv);
    int ng = num_groups, gsz = group_size, nh = num_heads, nkv = num_kv_heads, cprr = cpr, bsz = block_size,
        ml = max_len;
    void *pargs[] = {&context_lens, &shared_lens, &shared_eff, &start_tok, &qs, &qvs, &ng, &gsz, &nh, &nkv,
                     &cprr, &bsz, &ml, &err_word};
    cudaError_t e = launch_dependent(reinterpret_cast<const void *>(&prefix_prep_kernel),
                                     dim3(static_cast<unsigned>(blocks)), dim3(256), pargs, 0, cs);
    if (e != cudaSuccess)
        return bad(PA_ERR_CUDA, "shared-prefix prep launch failed");

    DecodeParams base;
    base.out = out;
    base.k_cache = k_cache;
    base.v_cache = v_cache;
    base.err = err_word;
    base.block_size = block_size;
    base.window = 0;
    base.max_len = max_len;
    base.num_blocks = num_blocks;
    base.bpp = pl.bpp;
    base.max_parts = pl.max_parts;
    base.out_dtype = out_dtype;
    base.stages = 0;
    base.scale_log2 = scale * 1.4426950408889634f;
    base.force_partial = 1;
    base.q_dtype = dtype;

    // 2) the shared prefix, once per group: one grouped "sequence" per group
    DecodeParams pre = base;
    pre.q = qv;
    pre.block_tables = block_tables;           // row g of the grouped view is row g * group_size
    pre.max_blocks_per_seq = max_blocks_per_seq * group_size;
    pre.context_lens = shared_eff;
    pre.start_tok = nullptr;
    pre.num_seqs = num_groups;
    pre.num_heads = num_kv_heads * Gp;
    pre.num_kv_heads = num_kv_heads;
    pre.part_acc = reinterpret_cast<float *>(ws + pl.pre_off);
    pre.part_ml = pre.part_acc + acc_floats;
    if (partition_size == 0) {
        // the prefix pass runs the tensor-core grouped-head kernel: its default
        // partition is twice as long (fewer partials; the region sized for the
        // shorter one holds them with its own row stride)
        pre.bpp = kGqaDefaultPartitionTokens / block_size;
        pre.max_parts = (pre.max_blocks_per_seq / group_size + pre.bpp - 1) / pre.bpp;
    }
    pa_status st = launch_decode_kernel(pre, dtype, head_dim, Gp, cs);
    if (st != PA_OK)
        return st;

    // 3) every sequence's own tokens after the prefix
    DecodeParams suf = base;
    suf.q = q;
    suf.block_tables = block_tables;
    suf.max_blocks_per_seq = max_blocks_per_seq;
    suf.context_lens = context_lens;
    suf.start_tok = start_tok;
    suf.num_seqs = num_seqs;
    suf.num_heads = num_heads;
    suf.num_kv_heads = num_kv_heads;
    suf.part_acc = reinterpret_cast<float *>(ws + pl.suf_off);
    suf.part_ml = suf.part_acc + acc_floats;
    st = launch_decode_kernel(suf, dtype, head_dim, G, cs);
    if (st != PA_OK)
        return st;

    // 4) merge
    const long long rows = static_cast<long long>(num_seqs) * num_heads;
    int gs = group_size;
    void *cargs[] = {&pre, &suf, &shared_eff, &gs};
    e = launch_dependent(reinterpret_cast<const void *>(&prefix_combine_kernel<128>),
                         dim3(static_cast<unsigned>((rows + kReduceRows - 1) / kReduceRows)), dim3(kReduceThreads),
                         cargs, 0, cs);
    if (e != cudaSuccess)
        return bad(PA_ERR_CUDA, "shared-prefix combine launch failed");
    return PA_OK;
}
