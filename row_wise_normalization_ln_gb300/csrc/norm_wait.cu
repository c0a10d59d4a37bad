// The ring kernels' bounded waits, per device: the time limit of a wait for
// a bulk copy and the count of CTAs whose wait gave up. Kernels read the
// limit and add to the count; the host sets the limit (norm_set_wait_limit),
// and reads and resets the count (norm_wait_timeouts, norm_synchronize).
#include <atomic>
#include <cstddef>

#include <cuda_runtime_api.h>

#include "libnorm.h"
#include "norm_args.h"

namespace {

// One per device. In host code the name is only a stand-in for the symbol:
// kernels get its device address from wait_state().
__device__ libnorm::WaitState g_wait = {0u, 0u, libnorm::kDefaultWaitLimitNs};

constexpr int kMaxDevices = 64;
std::atomic<libnorm::WaitState*> g_state[kMaxDevices] = {};

norm_status cuda_failed(cudaError_t e) {
    libnorm::note_cuda_error(static_cast<int>(e));
    return NORM_ERR_CUDA;
}

// Reads the current device's count and resets it to 0, after the device
// has finished all its work.
norm_status take_count(unsigned int* n) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbol(n, g_wait, sizeof(*n), offsetof(libnorm::WaitState, timeouts));
    const unsigned int zero = 0;
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_wait, &zero, sizeof(zero), offsetof(libnorm::WaitState, timeouts));
    return e == cudaSuccess ? NORM_OK : cuda_failed(e);
}

}  // namespace

namespace libnorm {

WaitState* wait_state(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    WaitState* p = g_state[dev].load(std::memory_order_acquire);
    if (p != nullptr) return p;
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_wait) != cudaSuccess) return nullptr;
    p = static_cast<WaitState*>(q);
    g_state[dev].store(p, std::memory_order_release);
    return p;
}

}  // namespace libnorm

extern "C" norm_status norm_wait_timeouts(uint32_t* count) {
    if (count == nullptr) return NORM_ERR_ARG;
    unsigned int n = 0;
    const norm_status st = take_count(&n);
    if (st != NORM_OK) return st;
    *count = n;
    return NORM_OK;
}

extern "C" norm_status norm_synchronize(void) {
    unsigned int n = 0;
    const norm_status st = take_count(&n);
    if (st != NORM_OK) return st;
    return n > 0 ? NORM_ERR_TIMEOUT : NORM_OK;
}

extern "C" norm_status norm_set_wait_limit(uint64_t ns) {
    if (ns > libnorm::kMaxWaitLimitNs) return NORM_ERR_ARG;
    const unsigned long long v = ns;
    const cudaError_t e = cudaMemcpyToSymbol(g_wait, &v, sizeof(v), offsetof(libnorm::WaitState, limit_ns));
    return e == cudaSuccess ? NORM_OK : cuda_failed(e);
}

extern "C" norm_status norm_wait_limit(uint64_t* ns) {
    if (ns == nullptr) return NORM_ERR_ARG;
    unsigned long long v = 0;
    const cudaError_t e = cudaMemcpyFromSymbol(&v, g_wait, sizeof(v), offsetof(libnorm::WaitState, limit_ns));
    if (e != cudaSuccess) return cuda_failed(e);
    *ns = v;
    return NORM_OK;
}
