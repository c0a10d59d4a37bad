// LayerNorm backward kernels, fp16 rows.
#include "norm_bwd.cuh"

namespace libnorm {

cudaError_t launch_ln_bwd_f16(const norm_plan& plan, const BwdArgs& a, cudaStream_t s, int dev, int num_sms) {
    return launch_norm_bwd<__half, true>(plan, a, s, dev, num_sms);
}

}  // namespace libnorm
