// MHA decode kernel instantiations for __nv_bfloat16 caches (head_dim 64/128, block 8/16/32).
#include "pa_decode_mha.cuh"
#include "pa_internal.h"

namespace pa {

const void *decode_mha_kernel_bf16(int head_dim, int block_size) {
#define PA_CASE(D, BS)                                                   \
    if (head_dim == D && block_size == BS)                               \
        return reinterpret_cast<const void *>(&pa_decode_mha_kernel<__nv_bfloat16, D, BS>);
    PA_CASE(64, 8) PA_CASE(64, 16) PA_CASE(64, 32)
    PA_CASE(128, 8) PA_CASE(128, 16) PA_CASE(128, 32)
#undef PA_CASE
    return nullptr;
}

}  // namespace pa
