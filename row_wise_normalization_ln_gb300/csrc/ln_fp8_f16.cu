// LayerNorm forward with an FP8 E4M3 output, fp16 rows: plain and with the
// fused residual add.
#include "norm_kernels.cuh"

namespace libnorm {

cudaError_t launch_ln_fp8_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev) {
    return launch_norm<__half, true, false, true>(plan, a, s, num_sms, dev);
}

cudaError_t launch_ln_add_fp8_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms,
                                     int dev) {
    return launch_norm<__half, true, true, true>(plan, a, s, num_sms, dev);
}

}  // namespace libnorm
