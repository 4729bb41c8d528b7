// pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
//
// pa_decode needs caller-provided scratch for the partial results of long
// contexts.  Some callers have no way to provide it: a plugin whose host
// framework owns every device allocation and forbids direct cudaMalloc, a
// runtime that works inside a fixed, pre-reserved memory budget, or a latency
// path that must not pay for an allocation (cudaMalloc can synchronise the
// device).  This entry point takes its scratch from one fixed array compiled
// into the library instead, so a call allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  All calls
// on a device share it and it keeps the previous call's contents; nothing in
// it has to start at zero (every partial the reduce kernel reads was written
// by the same call's decode kernel first).  Two calls whose work overlaps on
// the GPU (different streams, no ordering between them) race on the array and
// may return wrong results: order such calls on one stream or use pa_decode
// with separate workspaces.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

// In host code this name is only a stand-in for the device array, not its
// address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
cudaError_t scratch_address(void **addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" size_t pa_decode_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

extern "C" pa_status pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                       const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                                       int num_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                                       int window, pa_dtype dtype, pa_dtype out_dtype, int max_blocks_per_seq,
                                       int num_blocks, int partition_size, uint32_t *err_word,
                                       pa_stream_t stream) {
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                                                 window, partition_size);
    if (need > kNoAllocScratchBytes) {
        // pa_decode without a workspace checks every other argument first and
        // launches nothing: a bad argument is reported as itself, and only a
        // valid call comes back as too large for the scratch
        const pa_status st = pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                                       num_kv_heads, head_dim, block_size, scale, window, dtype, out_dtype,
                                       max_blocks_per_seq, num_blocks, partition_size, nullptr, 0, err_word, stream);
        if (st != PA_ERR_WORKSPACE_TOO_SMALL)
            return st;
        const std::string why = "pa_decode_noalloc needs " + std::to_string(need) +
                                " bytes of scratch for this shape; its built-in scratch holds " +
                                std::to_string(kNoAllocScratchBytes) +
                                " bytes (use pa_decode with a caller workspace, or a larger partition_size)";
        pa::set_last_error_detail(why.c_str());
        return PA_ERR_WORKSPACE_TOO_SMALL;
    }
    void *scratch = nullptr;
    if (need > 0) {
        const cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess) {
            const std::string why = std::string("pa_decode_noalloc scratch lookup: ") + cudaGetErrorName(e);
            pa::set_last_error_detail(why.c_str());
            return PA_ERR_CUDA;
        }
    }
    return pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, num_kv_heads,
                     head_dim, block_size, scale, window, dtype, out_dtype, max_blocks_per_seq, num_blocks,
                     partition_size, scratch, need > 0 ? kNoAllocScratchBytes : 0, err_word, stream);
}
