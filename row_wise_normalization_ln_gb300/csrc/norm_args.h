// Kernel argument block and per-(op, dtype) launchers shared by the host
// library and the kernel translation units. Host-visible only: no device code.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#include "libnorm.h"

namespace libnorm {

struct NormArgs {
    const void* x;      // [M, N]
    const void* gamma;  // [N] (LayerNorm gamma, RMSNorm w)
    const void* beta;   // [N] (LayerNorm only)
    void* y;            // [M, N]
    float* mean;        // [M] or null (LayerNorm only)
    float* rstd;        // [M] or null (LayerNorm only)
    int64_t M;
    int32_t N;
    float eps;
    int32_t group;      // GROUP mapping: lanes per row
    int32_t rounds;     // CTA mapping: register-sized rounds per row
};

// Launch the kernel variant `plan` names. The plan has been validated.
cudaError_t launch_ln_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s);
cudaError_t launch_ln_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s);
cudaError_t launch_rms_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s);
cudaError_t launch_rms_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s);

}  // namespace libnorm
