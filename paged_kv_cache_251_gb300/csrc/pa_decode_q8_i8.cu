// 8-bit-cache decode kernel instantiations (i8 codes; head_dim 64/128, group 1/2/4/8).
#include "pa_decode_q8.cuh"
#include "pa_internal.h"

namespace pa {

const void *decode_q8_kernel_i8(int head_dim, int group) {
#define PA_CASE(D, G)                     \
    if (head_dim == D && group == G)      \
        return reinterpret_cast<const void *>(&pa_decode_q8_kernel<kFmtI8, D, G>);
    PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
    PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
#undef PA_CASE
    return nullptr;
}

}  // namespace pa
