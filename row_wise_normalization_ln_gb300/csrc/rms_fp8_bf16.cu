// RMSNorm forward with an FP8 E4M3 output, bf16 rows: plain and with the
// fused residual add.
#include "norm_kernels.cuh"

namespace libnorm {

cudaError_t launch_rms_fp8_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev) {
    return launch_norm<__nv_bfloat16, false, false, true>(plan, a, s, num_sms, dev);
}

cudaError_t launch_rms_add_fp8_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms,
                                     int dev) {
    return launch_norm<__nv_bfloat16, false, true, true>(plan, a, s, num_sms, dev);
}

}  // namespace libnorm
