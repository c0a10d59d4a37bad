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
    int32_t stages;     // pipelined CTA mapping: shared-memory ring stages
};

// Launch the kernel variant `plan` names on the current device `dev` (with
// `num_sms` SMs). The plan has been validated; a pipelined plan with grid 0
// gets a persistent grid sized by occupancy.
cudaError_t launch_ln_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);

}  // namespace libnorm
