// Fused residual add + LayerNorm forward kernels, fp16 rows.
#include "norm_kernels.cuh"

namespace libnorm {

cudaError_t launch_ln_add_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev) {
    return launch_norm<__half, true, true>(plan, a, s, num_sms, dev);
}

}  // namespace libnorm
