// LayerNorm forward kernels, fp16 rows: every (mapping, access width,
// accesses per thread) variant the planner can name.
#include "norm_kernels.cuh"

namespace libnorm {

cudaError_t launch_ln_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev) {
    return launch_norm<__half, true, false>(plan, a, s, num_sms, dev);
}

}  // namespace libnorm
