// Internal interfaces between the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

struct DecodeParams;

// Launch `fn` so that it may be scheduled while the kernel before it on
// `stream` still runs (programmatic stream serialization; that kernel signals
// launch_dependents).  `fn` must execute griddepcontrol.wait before it reads
// anything the earlier kernel writes.
inline cudaError_t launch_dependent(const void *fn, dim3 grid, dim3 block, void **args, size_t smem,
                                    cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Decode kernel entry (as a function pointer for cudaLaunchKernel) for one
// element type, head_dim and query-group size; nullptr if not built.
const void *decode_kernel_f32(int head_dim, int group);
const void *decode_kernel_f16(int head_dim, int group);
const void *decode_kernel_bf16(int head_dim, int group);
const void *reduce_kernel(int head_dim);

// MHA (one query head per kv head) decode kernels fed by TMA tensor copies,
// per element type, head_dim and block size; nullptr if not built.
const void *decode_mha_kernel_f32(int head_dim, int block_size);
const void *decode_mha_kernel_f16(int head_dim, int block_size);
const void *decode_mha_kernel_bf16(int head_dim, int block_size);

// Tensor-core (tcgen05) decode kernels for grouped-query heads: 16-bit K/V,
// head_dim 128, per block size and group 2/4/8; nullptr if not built.
const void *decode_gqa_kernel_f16(int block_size, int group);
const void *decode_gqa_kernel_bf16(int block_size, int group);

// General decode kernels for 8-bit caches (INT8 / E4M3 codes with row
// scales), per head_dim and query group; nullptr if not built.
const void *decode_q8_kernel_i8(int head_dim, int group);
const void *decode_q8_kernel_e4m3(int head_dim, int group);

// Fast decode kernels for 8-bit caches fed by TMA tensor copies: head_dim
// 128, per query group (1, 2, 4) and block size; nullptr if not built.
const void *decode_q8f_kernel_i8(int group, int block_size);
const void *decode_q8f_kernel_e4m3(int group, int block_size);

// Tensor-core decode kernels for E4M3 pages (kind::f8f6f4): head_dim 128, 4 kv
// heads per item, per query group (2, 4) and block size (16, 32);
// nullptr if not built.
const void *decode_q8t_kernel_e4m3(int group, int block_size);
// A zeroed {next item, CTAs done} counter pair for one launch on `device` of
// a kernel that claims its items (the launch returns it to zero); nullptr if
// unavailable.
unsigned int *work_counter(int device, cudaStream_t stream);

cudaError_t launch_append(const void *k, const void *v, const int64_t *slots, void *k_cache, void *v_cache,
                          int num_tokens, int num_kv_heads, int row_bytes, int block_size, int num_blocks,
                          uint32_t *err, int num_sms, cudaStream_t stream);

cudaError_t launch_append_quant(const void *k, const void *v, const int64_t *slots, void *k_pages, void *v_pages,
                                int num_tokens, int num_kv_heads, int head_dim, int in_dtype, int cache_dtype,
                                int block_size, int num_blocks, uint32_t *err, int num_sms, cudaStream_t stream);

cudaError_t launch_copy_blocks(const int64_t *pairs, int num_pairs, void *k_cache, void *v_cache,
                               long long block_bytes, int num_blocks, uint32_t *err, int num_sms,
                               cudaStream_t stream);

cudaError_t launch_swap_blocks(const int64_t *pairs, int num_pairs, const void *src_k, const void *src_v,
                               void *dst_k, void *dst_v, long long block_bytes, int src_blocks, int dst_blocks,
                               uint32_t *err, int num_sms, cudaStream_t stream);

// Choose the decode kernel for (dtype, head_dim, group G, block size), encode
// its tensor maps and launch it on `cs` with the filled-in parameters (the
// stage count is set there).  The partition reduce is the caller's.
pa_status launch_decode_kernel(DecodeParams &p, int dtype, int head_dim, int G, cudaStream_t cs);

// Same for an 8-bit cache of cache_dtype (PA_I8 / PA_E4M3) in pages
// (pa_quant.cuh); p.q_dtype must be set.
pa_status launch_decode_q8_kernel(DecodeParams &p, int cache_dtype, int head_dim, int G, cudaStream_t cs);

// Text returned by pa_last_error_detail() on the calling thread.
void set_last_error_detail(const char *why);

}  // namespace pa
