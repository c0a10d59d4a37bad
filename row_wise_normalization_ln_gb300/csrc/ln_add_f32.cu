// Fused residual add + LayerNorm forward kernels, f32 rows.
#include "norm_kernels.cuh"

namespace libnorm {

cudaError_t launch_ln_add_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev) {
    return launch_norm<float, true, true>(plan, a, s, num_sms, dev);
}

}  // namespace libnorm
