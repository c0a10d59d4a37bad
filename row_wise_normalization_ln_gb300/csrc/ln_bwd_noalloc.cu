// ln_bwd_noalloc: the LayerNorm backward for callers that cannot allocate
// device memory. The column-gradient partial rows, which ln_bwd keeps in a
// workspace the caller provides, live here in one fixed-size static device
// array instead; the call then runs the same planned backward as
// ln_bwd_planned, with its grid capped so that the partial rows fit.
#include <cstdint>
#include <mutex>

#include <cuda_runtime_api.h>

#include "libnorm.h"
#include "norm_args.h"

namespace {

// 4 MiB of scratch. Every device that loads this library holds it until the
// process exits.
constexpr size_t kScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_scratch[kScratchFloats];

// Device address of g_scratch and SM count, per device, looked up once per
// device and process (a cudaDeviceReset while the library is loaded is not
// supported). In host code the name g_scratch is only a stand-in for the
// symbol, never a device address.
struct DeviceScratch {
    float* ptr;
    int sms;
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices] = {};

norm_status scratch_for_current_device(float** ptr, int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        libnorm::note_cuda_error(static_cast<int>(e));
        return NORM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return NORM_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_dev[dev].ptr == nullptr) {
        // First call on this device (which is current): look the array up once.
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || p == nullptr) {
            libnorm::note_cuda_error(static_cast<int>(e != cudaSuccess ? e : cudaErrorInvalidSymbol));
            return NORM_ERR_CUDA;
        }
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess || n <= 0) {
            libnorm::note_cuda_error(static_cast<int>(e));
            return NORM_ERR_CUDA;
        }
        g_dev[dev].ptr = static_cast<float*>(p);
        g_dev[dev].sms = n;
    }
    *ptr = g_dev[dev].ptr;
    *sms = g_dev[dev].sms;
    return NORM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" norm_status ln_bwd_noalloc(const void* dy, const void* x, const void* gamma, const float* mean,
                                      const float* rstd, void* dx, float* dgamma, float* dbeta, int64_t M,
                                      int64_t N, norm_dtype dtype, cudaStream_t stream) {
    const int al = aligned16(dy) && aligned16(x) && aligned16(gamma) && aligned16(dx);
    // Every argument check on the host before any CUDA call: the pointers
    // ln_bwd requires, the backward's own size limits, then the scratch
    // limit (one partial row of dgamma and dbeta must fit; the backward
    // refuses every N for which this guard could fail, so it only states the
    // array's bound).
    if (!dgamma || !dbeta) return NORM_ERR_ARG;
    if (M > 0 && (!dy || !x || !gamma || !dx || !mean || !rstd)) return NORM_ERR_ARG;
    norm_plan plan;
    norm_status st = norm_bwd_make_plan(M, N, dtype, 1, al, 1, &plan);
    if (st != NORM_OK) return st;
    if (static_cast<size_t>(2 * N) > kScratchFloats) return NORM_ERR_ARG;
    float* scratch = nullptr;
    int sms = 0;
    st = scratch_for_current_device(&scratch, &sms);
    if (st != NORM_OK) return st;
    st = norm_bwd_make_plan(M, N, dtype, 1, al, sms, &plan);
    if (st != NORM_OK) return st;
    // At most as many partial rows (grid / group) as the scratch holds: where
    // one partial row per CTA would not fit, CTAs of one row each first add
    // their columns in reduction clusters of up to 8, then the grid is capped.
    const int64_t rows_fit = static_cast<int64_t>(kScratchFloats / static_cast<size_t>(2 * N));
    if (plan.cluster == 1) {
        while (plan.grid / plan.group > rows_fit && plan.group < 8 && plan.group * 2 <= plan.grid) plan.group *= 2;
        plan.grid -= plan.grid % plan.group;
    }
    const int64_t cap = rows_fit * plan.group;
    if (plan.grid > cap) plan.grid = cap;
    return ln_bwd_planned(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, scratch, kScratchFloats * sizeof(float), M, N,
                          dtype, stream, &plan);
}
