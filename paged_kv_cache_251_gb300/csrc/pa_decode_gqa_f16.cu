// Tensor-core GQA decode kernel instantiations for __half caches (head_dim 128,
// block 8/16/32, query groups 2/4/8).
#include "pa_decode_gqa.cuh"
#include "pa_internal.h"

namespace pa {

const void *decode_gqa_kernel_f16(int block_size, int group) {
#define PA_CASE(BS, G)                                                   \
    if (block_size == BS && group == G)                                  \
        return reinterpret_cast<const void *>(&pa_decode_gqa_kernel<__half, BS, G>);
    PA_CASE(8, 2) PA_CASE(8, 4) PA_CASE(8, 8)
    PA_CASE(16, 2) PA_CASE(16, 4) PA_CASE(16, 8)
    PA_CASE(32, 2) PA_CASE(32, 4) PA_CASE(32, 8)
#undef PA_CASE
    return nullptr;
}

}  // namespace pa
