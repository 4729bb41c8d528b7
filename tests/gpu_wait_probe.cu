// Test helper, compiled by tests/test_gpu_failure.py: one CTA waits on an
// mbarrier that nothing arrives on, through the bounded wait every decode
// kernel uses (pa_device.cuh), and reports whether the wait gave up and after
// how long.  No fault, trap or endless loop: the wait ends by its time limit.
#include <cuda_runtime.h>

#include "pa_device.cuh"

namespace {

__global__ void wait_probe_kernel(unsigned int *status, unsigned long long *elapsed_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        pa::mbar_init(&bar, 1);
        pa::fence_mbar_init();
    }
    __syncthreads();
    const uint64_t t0 = pa::globaltimer_ns();
    const bool completed = pa::mbar_wait_bounded(&bar, 0);  // phase 0: no thread ever arrives
    const uint64_t t1 = pa::globaltimer_ns();
    if (threadIdx.x == 0) {
        *status = completed ? 1u : 2u;
        *elapsed_ns = t1 - t0;
    }
}

}  // namespace

// 0 on success, with *status = 2 when the wait gave up (1: it completed).
extern "C" int wait_probe_run(unsigned int *status, unsigned long long *elapsed_ns) {
    unsigned int *d_status = nullptr;
    unsigned long long *d_elapsed = nullptr;
    if (cudaMalloc(&d_status, sizeof(unsigned int)) != cudaSuccess)
        return 1;
    if (cudaMalloc(&d_elapsed, sizeof(unsigned long long)) != cudaSuccess) {
        cudaFree(d_status);
        return 1;
    }
    wait_probe_kernel<<<1, 32>>>(d_status, d_elapsed);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(status, d_status, sizeof(unsigned int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
        e = cudaMemcpy(elapsed_ns, d_elapsed, sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(d_status);
    cudaFree(d_elapsed);
    return e == cudaSuccess ? 0 : 2;
}
