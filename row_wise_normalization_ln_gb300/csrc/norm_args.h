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

// Per-device state of the ring kernels' bounded waits (one instance per
// device, in device memory): the count of CTAs whose wait for a bulk copy
// gave up, and the time limit of the per-row waits. The host reads and
// resets the count (norm_wait_timeouts, norm_synchronize) and sets the limit
// (norm_set_wait_limit).
struct WaitState {
    unsigned int timeouts;
    unsigned int pad;
    unsigned long long limit_ns;
};

// Default limit of a per-row wait, and the fixed limit of the waits a CTA
// makes before it exits for copies still in flight (those always get the
// full time, so that no copy lands in the shared memory of a CTA that has
// gone).
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
constexpr unsigned long long kMaxWaitLimitNs = 60000000000ull;

struct NormArgs {
    const void* x;      // [M, N], row pitch ldx
    const void* gamma;  // [N] (LayerNorm gamma, RMSNorm w)
    const void* beta;   // [N] (LayerNorm only)
    void* y;            // [M, N], row pitch ldy
    float* mean;        // [M] or null (LayerNorm only)
    float* rstd;        // [M] or null (LayerNorm only)
    const void* res;    // [M, N] residual (fused residual add only)
    void* h;            // [M, N] h = x + res (fused residual add only)
    const float* qscale;  // FP8 output only: the static scale (y is then uint8 E4M3 codes)
    int64_t M;
    int32_t N;
    float eps;
    int32_t group;      // GROUP mapping: lanes per row; CTA mapping: L2 prefetch of the row group-1 ahead (0: none)
    int32_t rounds;     // CTA mapping: register-sized rounds per row
    int32_t stages;     // ring CTA mapping: shared-memory stages
    int16_t shift = 0;       // CTA mapping, 16-byte vectors: rows need not start on a 16-byte boundary
    int16_t vec_params = 1;  // gamma (and beta) 16-byte aligned
    int64_t ldx = 0;         // row pitch of x in elements (set to N for contiguous rows)
    int64_t ldy = 0;         // row pitch of y in elements (bytes for an FP8 y)
    WaitState* wait = nullptr;  // ring kernels: this device's wait limit and count of waits that gave up
};
// Kept at 128 bytes: a larger argument block made ptxas spill the 64-register
// long-row kernels.
static_assert(sizeof(NormArgs) == 128, "kernel argument block: 128 bytes");

// Backward pass. A CTA (row_cluster == 1) or a cluster of row_cluster CTAs
// owns one row at a time; each thread accumulates the column gradients of
// its own columns over the rows it visits. Those accumulators leave through
// `ws` as partial rows [partials][narr][N] (narr = 2 for LayerNorm: dgamma,
// dbeta; 1 for RMSNorm: dw), which a second kernel sums in a fixed order.
struct BwdArgs {
    const void* dy;       // [M, N]
    const void* x;        // [M, N]
    const void* gamma;    // [N] (LayerNorm gamma, RMSNorm w)
    const float* mean;    // [M] (LayerNorm)
    const float* rstd;    // [M] (LayerNorm)
    void* dx;             // [M, N]
    float* ws;            // [partials][narr][N]
    float* dgamma;        // [N] (LayerNorm dgamma, RMSNorm dw)
    float* dbeta;         // [N] (LayerNorm)
    int64_t M;
    int32_t N;
    float eps;            // RMSNorm (rstd is recomputed from x)
    int32_t row_cluster;  // CTAs per row
    int32_t stages = 0;   // 1: register pipeline; 2..4: shared-memory stages of upcoming rows; 0: neither
    WaitState* wait = nullptr;  // ring and pipeline kernels: this device's wait limit and count of waits that gave up
};

constexpr int kBwdMaxThreads = 512;

// Record a CUDA error for norm_last_cuda_error() on the calling thread.
void note_cuda_error(int e);

// CTA size limit of the ring kernels: a thread holds its elements widened to
// fp32, up to 64 registers of them.
constexpr int kRingMaxThreads = 512;

// Dynamic shared memory of a forward ring launch: the stages' 16-byte
// slots, then one 16-byte slot (the row's first 16 bytes) and one 8-byte
// mbarrier per stage.
inline int64_t ring_smem_bytes(int stages, int per_thread, int threads) {
    return int64_t(stages) * (int64_t(per_thread) * threads * 16 + 16 + 8);
}

// Device address of the current device's WaitState (the ring kernels' wait
// limit and count); null if it cannot be resolved.
WaitState* wait_state(int dev);

// Dynamic shared memory of a backward launch: the column accumulators
// ([2 for LayerNorm | 1][threads * per_thread * vec] fp32) and, for a ring
// (stages >= 2), per stage two slices of 16-byte slots (x, dy) and an 8-byte
// mbarrier: after the accumulators, or over them when those stay in
// registers until the last row.
inline int64_t bwd_smem_bytes(bool ln, int threads, int per_thread, int vec, int stages) {
    const int64_t acc = int64_t(ln ? 2 : 1) * threads * per_thread * vec * 4;
    if (stages < 2) return acc;  // stages 1, the register pipeline, keeps no rows here
    const int64_t ring = int64_t(stages) * (2 * int64_t(threads) * per_thread * 16 + 8);
    // Accumulators held in registers until the end (all but the 16-bit
    // variants of 4 accesses per thread) share their slots with the ring.
    const bool acc_in_registers = !(vec == 8 && per_thread >= 4);
    return acc_in_registers ? (acc > ring ? acc : ring) : acc + ring;
}

// Partial rows of the column gradients a backward plan produces (one per
// cluster, or per CTA without clusters).
inline int64_t bwd_partials(const norm_plan& p) { return p.group > 0 ? p.grid / p.group : 0; }

cudaError_t launch_ln_bwd_f32(const norm_plan& plan, const BwdArgs& a, cudaStream_t s, int dev, int num_sms);
cudaError_t launch_ln_bwd_bf16(const norm_plan& plan, const BwdArgs& a, cudaStream_t s, int dev, int num_sms);
cudaError_t launch_rms_bwd_f32(const norm_plan& plan, const BwdArgs& a, cudaStream_t s, int dev, int num_sms);
cudaError_t launch_rms_bwd_bf16(const norm_plan& plan, const BwdArgs& a, cudaStream_t s, int dev, int num_sms);
cudaError_t launch_ln_bwd_f16(const norm_plan& plan, const BwdArgs& a, cudaStream_t s, int dev, int num_sms);
cudaError_t launch_rms_bwd_f16(const norm_plan& plan, const BwdArgs& a, cudaStream_t s, int dev, int num_sms);

// Launch the kernel variant `plan` names on the current device `dev` (with
// `num_sms` SMs). The plan has been validated; a ring plan with grid 0
// gets a persistent grid sized by occupancy.
cudaError_t launch_ln_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
// FP8 E4M3 output (a.qscale set; y holds one byte per element), without and
// with the fused residual add.
cudaError_t launch_ln_fp8_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_fp8_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_fp8_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_fp8_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_fp8_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_fp8_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_add_fp8_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_add_fp8_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_add_fp8_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_add_fp8_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_add_fp8_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_add_fp8_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
// The same with the fused residual add (a.res, a.h set).
cudaError_t launch_ln_add_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_add_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_add_f32(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_add_bf16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_ln_add_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);
cudaError_t launch_rms_add_f16(const norm_plan& plan, const NormArgs& a, cudaStream_t s, int num_sms, int dev);

}  // namespace libnorm
