// The device counter of ring-kernel waits that gave up: a bulk copy that
// did not complete within the wait's limit. Kernels add to it; the host
// reads and resets it with norm_wait_timeouts.
#include <atomic>

#include <cuda_runtime_api.h>

#include "libnorm.h"
#include "norm_args.h"

namespace {

__device__ unsigned int g_wait_timeouts;  // one per device

constexpr int kMaxDevices = 64;
std::atomic<unsigned int*> g_counter[kMaxDevices] = {};

}  // namespace

namespace libnorm {

unsigned int* wait_counter(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned int* p = g_counter[dev].load(std::memory_order_acquire);
    if (p != nullptr) return p;
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_wait_timeouts) != cudaSuccess) return nullptr;
    p = static_cast<unsigned int*>(q);
    g_counter[dev].store(p, std::memory_order_release);
    return p;
}

}  // namespace libnorm

extern "C" norm_status norm_wait_timeouts(uint32_t* count) {
    if (count == nullptr) return NORM_ERR_ARG;
    unsigned int n = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&n, g_wait_timeouts, sizeof(n));
    const unsigned int zero = 0;
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(zero));
    if (e != cudaSuccess) {
        libnorm::note_cuda_error(static_cast<int>(e));
        return NORM_ERR_CUDA;
    }
    *count = n;
    return NORM_OK;
}
