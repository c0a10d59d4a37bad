// Kernel argument block and per-(op, dtype) launchers shared by the host
// library and the kernel translation units. Host-visible only: no device code.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#include "libnorm.h"

namespace libnorm {

// CTA size limit of the fused residual-add kernels: x and the residual are in
// flight together, which needs more than the 64 registers a 1024-thread CTA
// leaves each thread.
constexpr int kFusedMaxThreads = 512;

struct NormArgs {
    const void* x;      // [M, N]
    const void* gamma;  // [N] (LayerNorm gamma, RMSNorm w)
    const void* beta;   // [N] (LayerNorm only)
    void* y;            // [M, N]
    float* mean;        // [M] or null (LayerNorm only)
    float* rstd;        // [M] or null (LayerNorm only)
    const void* res;    // [M, N] residual (fused residual add only)
    void* h;            // [M, N] h = x + res (fused residual add only)
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
// The same with the fused residual add (a.res, a.h set).
cudaError_t launch_ln_add_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_add_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_add_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_add_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);

}  // namespace libnorm
