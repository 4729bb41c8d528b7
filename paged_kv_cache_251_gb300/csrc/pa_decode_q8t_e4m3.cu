// Tensor-core decode over E4M3 pages: instantiations (head_dim 128, block
// size 16 / 32, 2 / 4 query heads per kv head).
#include <atomic>
#include <mutex>

#include "pa_decode_q8t.cuh"
#include "pa_internal.h"

namespace pa {

// Item counters for dynamic scheduling: zero when the module loads, and every
// launch returns its pair to zero.  Launches take pairs round-robin, so
// launches in flight at the same time (up to kWorkSlots) never share one.
constexpr int kWorkSlots = 4096;
constexpr int kMaxDevices = 64;
__device__ unsigned int g_q8t_work[2 * kWorkSlots];

unsigned int *q8t_work_counter(int device) {
    static unsigned int *base[kMaxDevices] = {};
    static std::mutex mu;
    static std::atomic<unsigned int> next{0};
    if (device < 0 || device >= kMaxDevices)
        return nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!base[device]) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_q8t_work) != cudaSuccess)
                return nullptr;
            base[device] = static_cast<unsigned int *>(ptr);
        }
    }
    return base[device] + 2 * (next.fetch_add(1u) % kWorkSlots);
}

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
