// Tensor-core decode over E4M3 pages: instantiations (head_dim 128, block
// size 16 / 32, 2 / 4 query heads per kv head).
#include "pa_decode_q8t.cuh"
#include "pa_internal.h"

namespace pa {

const void *decode_q8t_kernel_e4m3(int group, int block_size) {
#define PA_CASE(BS, G)                          \
    if (block_size == BS && group == G)         \
        return reinterpret_cast<const void *>(&pa_decode_q8t_kernel<BS, G>);
    PA_CASE(16, 2) PA_CASE(16, 4)
    PA_CASE(32, 2) PA_CASE(32, 4)
#undef PA_CASE
    return nullptr;
}

}  // namespace pa
