// Fast 8-bit-cache decode kernel instantiations (i8 codes; head_dim 128, group 1/2/4, block 8/16/32).
#include "pa_decode_q8f.cuh"
#include "pa_internal.h"

namespace pa {

const void *decode_q8f_kernel_i8(int group, int block_size) {
#define PA_CASE(G, BS)                              \
    if (group == G && block_size == BS)             \
        return reinterpret_cast<const void *>(&pa_decode_q8f_kernel<kFmtI8, G, BS>);
    PA_CASE(1, 8) PA_CASE(1, 16) PA_CASE(1, 32)
    PA_CASE(2, 8) PA_CASE(2, 16) PA_CASE(2, 32)
    PA_CASE(4, 8) PA_CASE(4, 16) PA_CASE(4, 32)
#undef PA_CASE
    return nullptr;
}

}  // namespace pa
