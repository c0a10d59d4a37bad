/*
 * libnorm - row-wise LayerNorm and RMSNorm forward for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (page title, section):
 *   [Ch7]  "第 7 章 LayerNorm 与 RMSNorm" (CUDA 算子工程): §7.1 LayerNorm
 *          definition, §7.4 Welford, §7.4.1 parallel merge, §7.5 RMSNorm,
 *          §7.6 fused kernel structure (per-row statistics, mean/rstd saved),
 *          §7.7 backward formulas, §7.9 FP8 output for the next GEMM.
 *   [RMS2] "CUDA算子优化(2)：RMSNorm": §1 formula, §2 [B*T, C] layout.
 *   [T3]   "T3 讲解：LayerNorm / RMSNorm 的 forward": §② masking, biased
 *          variance, fp32 statistics; §④ host reshape to [M, N]; §⑤ fusion
 *          with the residual add.
 *
 * Conventions shared by every entry point:
 *   - All pointers are DEVICE pointers on the current CUDA device, owned by
 *     the caller. The library allocates nothing and keeps no state between
 *     calls (the backward's scratch is a caller-provided workspace); work is enqueued asynchronously on `stream` (NULL = the legacy
 *     default stream). The caller keeps buffers alive until the stream has
 *     finished the call.
 *   - x and y are [M, N] row-major and contiguous (row stride N elements).
 *     gamma, beta and w are [N]. x, y, gamma, beta and w all have the element
 *     type `dtype`; mean and rstd are always fp32 [M] ([T3] §⑥).
 *   - Statistics and all arithmetic are fp32; bf16 and fp16 inputs are
 *     widened exactly and bf16 and fp16 outputs are rounded to nearest-even
 *     (fp16 outputs beyond its range become infinities).
 *   - y may equal x exactly (in place). Any other overlap between outputs and
 *     inputs, or between outputs, is undefined.
 *   - Pointers need no particular alignment beyond their element type.
 *     When x, y and the parameter vectors are 16-byte aligned and a row is a
 *     multiple of 16 bytes, the kernels use 128-bit accesses throughout.
 *     When the row tensors (x, y; with the fused add also residual and h)
 *     merely share their offset within 16 bytes (odd N, or tensors that
 *     start at the same misalignment), rows of 64 or more vectors still use
 *     128-bit accesses from each row's first aligned element, with the few
 *     elements before and after taken one by one (gamma and beta then by
 *     element where their vectors are not aligned). Otherwise the kernels
 *     use element accesses.
 *   - Argument errors are detected on the host before any CUDA call and
 *     nothing is launched. M == 0 is a no-op that returns NORM_OK (pointers
 *     may then be NULL). Limits: 1 <= N <= 2^24 (the largest count fp32
 *     holds exactly, [Ch7] §7.8), M >= 0, M*N < 2^63, eps finite and >= 0.
 *   - A CUDA error during the device query or the launch returns
 *     NORM_ERR_CUDA; norm_last_cuda_error() then gives the cudaError_t.
 */
#ifndef LIBNORM_H
#define LIBNORM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { NORM_F32 = 0, NORM_BF16 = 1, NORM_F16 = 2 } norm_dtype;

typedef enum {
    NORM_OK = 0,
    NORM_ERR_ARG = -1,    /* bad size, NULL pointer or eps */
    NORM_ERR_DTYPE = -2,  /* dtype not one of norm_dtype */
    NORM_ERR_CUDA = -3,   /* CUDA runtime error (device query or launch) */
    NORM_ERR_PLAN = -4,   /* an explicit plan is inconsistent with the call */
    NORM_ERR_TIMEOUT = -5 /* norm_synchronize: a ring kernel's wait for a
                             bulk copy ran out; those calls' outputs are void */
} norm_status;

/* How rows map onto the GPU. */
typedef enum {
    NORM_MAP_GROUP = 0,   /* `group` lanes of a warp own one row; a CTA of
                             `threads` threads holds threads/group rows */
    NORM_MAP_CTA = 1      /* `cluster` CTAs of `threads` threads own one row;
                             statistics meet in shared memory, and across the
                             cluster in distributed shared memory */
} norm_mapping;

/*
 * A launch plan. Each thread keeps `per_thread` accesses of `vec_elems`
 * elements of its row in registers. If one pass of the row's owners cannot
 * hold the whole row (CTA mapping only), the row is walked in `rounds`
 * register-sized rounds: x is read once for the statistics and the earlier
 * rounds are read again for the output (served from L2 when they fit).
 *
 * With `stages` >= 2 (CTA mapping, 16-byte vectors, one round) the CTAs are
 * persistent and keep up to `stages` upcoming rows of their share in flight
 * in a ring of shared-memory stages (one bulk copy per CTA and row) while
 * they reduce and store the current row; each thread widens its elements
 * to fp32 once. `grid` 0 then means "as many CTAs as fit on the device",
 * resolved at launch from the kernel's occupancy.
 */
typedef struct {
    int32_t mapping;     /* norm_mapping */
    int32_t vec_elems;   /* elements per access: 16/sizeof(element) or 1 */
    int32_t per_thread;  /* accesses per thread per round: 1, 2, 4 or 8 */
    int32_t group;       /* GROUP mapping: lanes per row, power of 2 <= 32 */
    int32_t threads;     /* threads per CTA, multiple of 32, <= 1024 */
    int32_t cluster;     /* CTA mapping: CTAs per row, 1, 2, 4 or 8 */
    int32_t rounds;      /* derived by norm_make_plan; ignored on input */
    int32_t stages;      /* 0: registers only; 2..4: shared-memory ring */
    int64_t grid;        /* CTAs launched (a multiple of `cluster`); rows
                            are walked in a grid-stride loop */
} norm_plan;

/*
 * LayerNorm forward ([Ch7] §7.1, §7.6; [T3] §②):
 *   mean_r = sum_i x_ri / N
 *   var_r  = sum_i (x_ri - mean_r)^2 / N        (biased, never E[x^2]-E[x]^2)
 *   rstd_r = 1 / sqrt(var_r + eps)
 *   y_ri   = (x_ri - mean_r) * rstd_r * gamma_i + beta_i
 * mean and rstd may each be NULL (not written). gamma and beta are required.
 */
norm_status ln_fwd(const void* x, const void* gamma, const void* beta, void* y,
                   float* mean, float* rstd, int64_t M, int64_t N, float eps,
                   norm_dtype dtype, cudaStream_t stream);

/*
 * RMSNorm forward ([Ch7] §7.5; [RMS2] §1; [T3] §③):
 *   rstd_r = 1 / sqrt(sum_i x_ri^2 / N + eps)
 *   y_ri   = x_ri * rstd_r * w_i
 * No statistics are written.
 */
norm_status rms_fwd(const void* x, const void* w, void* y, int64_t M, int64_t N,
                    float eps, norm_dtype dtype, cudaStream_t stream);

/*
 * The plan ln_fwd / rms_fwd would choose for M rows of N elements of
 * `dtype` on a device with `num_sms` SMs. `aligned16`: 1 when every pointer
 * is 16-byte aligned, 2 when the row tensors (x, y, and residual and h when
 * fused) only share their offset within 16 bytes (or rows are not whole
 * vectors), 0 otherwise (element accesses). Host only: makes no CUDA call.
 * Fills `plan` (including `rounds`) and returns NORM_OK, or an argument
 * error.
 */
norm_status norm_make_plan(int64_t M, int64_t N, norm_dtype dtype, int aligned16,
                           int num_sms, norm_plan* plan);

/*
 * ln_fwd / rms_fwd with an explicit plan (plan == NULL: choose as the plain
 * calls do). The plan is checked against the call on the host; a plan whose
 * accesses would not cover the row, whose vector width does not match the
 * dtype and alignment, whose ring would not fit in 227 KB of shared memory,
 * or whose shape is out of range returns NORM_ERR_PLAN and launches nothing.
 * For tuning and for tests of every kernel variant.
 */
norm_status ln_fwd_planned(const void* x, const void* gamma, const void* beta, void* y,
                           float* mean, float* rstd, int64_t M, int64_t N, float eps,
                           norm_dtype dtype, cudaStream_t stream, const norm_plan* plan);

norm_status rms_fwd_planned(const void* x, const void* w, void* y, int64_t M, int64_t N,
                            float eps, norm_dtype dtype, cudaStream_t stream,
                            const norm_plan* plan);

/*
 * ln_fwd / rms_fwd on strided rows ([T3] §④: the host wrapper keeps a
 * row-strided view and copies only when the innermost stride is not 1):
 * row r of x starts at x + r * ldx and row r of y at y + r * ldy (pitches in
 * elements, each >= N), e.g. a column block of a wider matrix. y may be x
 * itself when ldy == ldx. `plan` may be NULL (the plan ln_fwd would choose);
 * otherwise it is checked as for ln_fwd_planned. Rows whose pitches differ
 * modulo 16 bytes, or that start at different offsets within 16 bytes, use
 * element accesses.
 */
norm_status ln_fwd_strided(const void* x, int64_t ldx, const void* gamma, const void* beta,
                           void* y, int64_t ldy, float* mean, float* rstd, int64_t M,
                           int64_t N, float eps, norm_dtype dtype, cudaStream_t stream,
                           const norm_plan* plan);

norm_status rms_fwd_strided(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy,
                            int64_t M, int64_t N, float eps, norm_dtype dtype,
                            cudaStream_t stream, const norm_plan* plan);

/*
 * Fused residual add + LayerNorm ([Ch7] §7.9-7.10, the add + norm of a
 * transformer's residual stream; [T3] §⑤):
 *   h_ri = x_ri + residual_ri, rounded to `dtype` (exactly what a separate
 *          add kernel would store)
 *   y, mean, rstd = ln_fwd of h
 * Reads x and residual once and writes h and y. residual and h are [M, N]
 * with the layout of x. h may be x or residual itself, and so may y (the
 * usual in-place residual update); h and y must be different buffers
 * (NORM_ERR_ARG otherwise). Any other overlap is undefined.
 */
norm_status ln_fwd_add(const void* x, const void* residual, const void* gamma,
                       const void* beta, void* h, void* y, float* mean, float* rstd,
                       int64_t M, int64_t N, float eps, norm_dtype dtype,
                       cudaStream_t stream);

/* Fused residual add + RMSNorm: h as for ln_fwd_add, y = rms_fwd of h. */
norm_status rms_fwd_add(const void* x, const void* residual, const void* w, void* h,
                        void* y, int64_t M, int64_t N, float eps, norm_dtype dtype,
                        cudaStream_t stream);

/* The plan ln_fwd_add / rms_fwd_add would choose: as norm_make_plan, with
 * CTAs of at most 512 threads (the fused kernels keep two loads per access
 * in flight and need the registers). `aligned16` as for norm_make_plan
 * (0, 1 or 2), over all six pointers. Host only. */
norm_status norm_make_plan_add(int64_t M, int64_t N, norm_dtype dtype, int aligned16,
                               int num_sms, norm_plan* plan);

/* The fused calls with an explicit plan, checked as for ln_fwd_planned;
 * plans with `stages` != 0 or more than 512 threads return NORM_ERR_PLAN. */
norm_status ln_fwd_add_planned(const void* x, const void* residual, const void* gamma,
                               const void* beta, void* h, void* y, float* mean,
                               float* rstd, int64_t M, int64_t N, float eps,
                               norm_dtype dtype, cudaStream_t stream,
                               const norm_plan* plan);

norm_status rms_fwd_add_planned(const void* x, const void* residual, const void* w,
                                void* h, void* y, int64_t M, int64_t N, float eps,
                                norm_dtype dtype, cudaStream_t stream,
                                const norm_plan* plan);

/*
 * LayerNorm backward ([Ch7] §7.7; [T3] §⑥: the forward's fp32 mean and rstd
 * are reused, so the backward makes no statistics pass of its own):
 *   xhat_ri = (x_ri - mean_r) * rstd_r,   g_ri = dy_ri * gamma_i
 *   dx_ri   = rstd_r * (g_ri - sum_j g_rj / N - xhat_ri * sum_j g_rj xhat_rj / N)
 *   dgamma_i = sum_r dy_ri * xhat_ri,     dbeta_i = sum_r dy_ri
 * dy, x, dx: [M, N] of `dtype`; gamma: [N] of `dtype`; mean, rstd: fp32 [M]
 * as written by ln_fwd; dgamma, dbeta: fp32 [N] (always written; zero when
 * M == 0). dx may be dy or x itself; any other overlap is undefined.
 * `workspace` (device memory owned by the caller, 16-byte aligned, at least
 * norm_bwd_workspace_bytes() for the plan norm_bwd_make_plan chooses on this
 * device; may be NULL when that is 0) holds the partial column sums; calls
 * sharing a workspace must not overlap on the GPU. The column sums are added
 * in a fixed order: results are deterministic for a given plan.
 * Limit: a row must fit one register pass of a cluster of 8 CTAs of 512
 * threads: N <= 65536 (fp32, bf16 LayerNorm) or 131072 (bf16 RMSNorm) with
 * 16-byte vectors, N <= 32768 with element accesses; longer rows return
 * NORM_ERR_ARG.
 */
norm_status ln_bwd(const void* dy, const void* x, const void* gamma, const float* mean,
                   const float* rstd, void* dx, float* dgamma, float* dbeta, void* workspace,
                   size_t workspace_bytes, int64_t M, int64_t N, norm_dtype dtype,
                   cudaStream_t stream);

/*
 * RMSNorm backward ([Ch7] §7.7, last paragraph: one row sum). rstd is
 * recomputed from x with `eps` (rms_fwd saves no statistics; x is in
 * registers, so this costs no memory traffic):
 *   rstd_r = 1 / sqrt(sum_j x_rj^2 / N + eps)
 *   dx_ri  = rstd_r * w_i * dy_ri - x_ri * rstd_r^3 * sum_j dy_rj w_j x_rj / N
 *   dw_i   = sum_r dy_ri * x_ri * rstd_r            (fp32 [N])
 * Layout, workspace, aliasing and limits as for ln_bwd.
 */
norm_status rms_bwd(const void* dy, const void* x, const void* w, void* dx, float* dw,
                    void* workspace, size_t workspace_bytes, int64_t M, int64_t N, float eps,
                    norm_dtype dtype, cudaStream_t stream);

/*
 * The backward plan for M rows of N elements (`layer_norm` != 0 for ln_bwd)
 * on a device with `num_sms` SMs; host only. In a backward plan `cluster`
 * CTAs cover a row in one pass (rounds = 1) and `group` is the launched
 * cluster size: equal to `cluster` when a row spans several CTAs, otherwise
 * the number of CTAs (each on its own rows) whose column sums are added in
 * distributed shared memory before one partial row goes to the workspace.
 * At most `grid` CTAs walk the rows in a grid-stride loop: the launch takes
 * no more than can be resident on the device at once (0 when M == 0).
 * `aligned16` != 0 when dy, x, gamma and dx are 16-byte aligned (the
 * backward has no shifted-row mode: other rows use element accesses).
 * `stages` 2..4 (16-byte vector rows): each CTA keeps its slices of x and dy
 * of that many upcoming rows in a shared-memory ring filled by bulk copies
 * (bounded waits, counted by norm_wait_timeouts); 1 (one CTA per row,
 * cluster == 1): the register pipeline, each thread loading the next row's
 * slices into a second set of registers while the current row is reduced
 * and written; 0: rows are read from L2 after a prefetch. The planner takes
 * 2 stages for fp32 vector rows and 1 for 16-bit vector rows of one CTA.
 * Returns NORM_ERR_ARG for rows beyond the backward's limit.
 */
norm_status norm_bwd_make_plan(int64_t M, int64_t N, norm_dtype dtype, int layer_norm,
                               int aligned16, int num_sms, norm_plan* plan);

/* Workspace bytes a backward plan needs: (grid / group) partial rows of N
 * fp32 values, two arrays for LayerNorm, one for RMSNorm. Host only. */
norm_status norm_bwd_workspace_bytes(const norm_plan* plan, int64_t N, int layer_norm,
                                     size_t* bytes);

/* The backward with an explicit plan (checked on the host as above;
 * NORM_ERR_PLAN if it does not fit the call). */
norm_status ln_bwd_planned(const void* dy, const void* x, const void* gamma, const float* mean,
                           const float* rstd, void* dx, float* dgamma, float* dbeta,
                           void* workspace, size_t workspace_bytes, int64_t M, int64_t N,
                           norm_dtype dtype, cudaStream_t stream, const norm_plan* plan);

norm_status rms_bwd_planned(const void* dy, const void* x, const void* w, void* dx, float* dw,
                            void* workspace, size_t workspace_bytes, int64_t M, int64_t N,
                            float eps, norm_dtype dtype, cudaStream_t stream,
                            const norm_plan* plan);

/*
 * ln_bwd for callers that cannot allocate device memory: the same result as
 * ln_bwd, with no workspace argument. (The source pages have no counterpart;
 * this is an interface convenience.) Such callers include inference and
 * training runtimes that plan all device memory up front and forbid any
 * allocation afterwards, code that cannot reach the framework's allocator,
 * and latency-critical loops that cannot afford the device-wide
 * synchronisation cudaFree may cause. The call allocates nothing: the
 * backward's partial column sums go to one static device array of 4 MiB,
 * which every GPU that loads this library holds until the process exits.
 * Where one partial row (2 * N floats) per CTA would not fit, CTAs of one
 * row each are grouped into reduction clusters of up to 8, and then the
 * plan's grid is capped so that its partial rows fit; a row whose single
 * partial row would not fit (N > 524288, beyond the backward's own limits
 * anyway) returns NORM_ERR_ARG, as do the sizes ln_bwd refuses.
 * The first call on each device looks up that array's device address (with
 * the device current) and the SM count; make that first call before any
 * stream capture. The address is kept for the life of the process: a
 * cudaDeviceReset while the library is loaded is not supported. Nothing in the array needs to start at zero: each call
 * writes every partial row before reading it. All calls on a device share
 * the array, so calls that overlap on the GPU (on different streams, or
 * from different threads) race and corrupt each other's column gradients:
 * serialise them.
 */
norm_status ln_bwd_noalloc(const void* dy, const void* x, const void* gamma, const float* mean,
                           const float* rstd, void* dx, float* dgamma, float* dbeta, int64_t M,
                           int64_t N, norm_dtype dtype, cudaStream_t stream);

/*
 * Norm with an FP8 output for the next GEMM ([Ch7] §7.9: the norm writes
 * the GEMM's quantised input itself, as vLLM's static-scale fused kernels
 * do, instead of writing y in high precision for a separate quantiser):
 *   y8_ri = E4M3(y_ri / scale)
 * with y as ln_fwd / rms_fwd compute it (in fp32), `scale` one fp32 value
 * in device memory (a per-tensor static scale), E4M3 the OCP FP8 format
 * (4 exponent, 3 fraction bits, finite only, largest 448) with
 * round-to-nearest-even and saturation: magnitudes from 448 give +-448.
 * y8 is [M, N] bytes (E4M3 codes), row stride N. mean and rstd as for
 * ln_fwd. The scale must be finite and nonzero (not checked: it is read on
 * the device). y8 may not overlap x.
 */
norm_status ln_fwd_fp8(const void* x, const void* gamma, const void* beta, const float* scale,
                       void* y8, float* mean, float* rstd, int64_t M, int64_t N, float eps,
                       norm_dtype dtype, cudaStream_t stream);

norm_status rms_fwd_fp8(const void* x, const void* w, const float* scale, void* y8, int64_t M,
                        int64_t N, float eps, norm_dtype dtype, cudaStream_t stream);

/* The fused residual add with an FP8 output: h as for ln_fwd_add (h may be
 * x or residual itself), y8 = E4M3(norm(h) / scale). */
norm_status ln_fwd_add_fp8(const void* x, const void* residual, const void* gamma,
                           const void* beta, const float* scale, void* h, void* y8, float* mean,
                           float* rstd, int64_t M, int64_t N, float eps, norm_dtype dtype,
                           cudaStream_t stream);

norm_status rms_fwd_add_fp8(const void* x, const void* residual, const void* w,
                            const float* scale, void* h, void* y8, int64_t M, int64_t N, float eps,
                            norm_dtype dtype, cudaStream_t stream);

/* The FP8-output calls with an explicit plan (residual == NULL: no fused
 * add, h ignored); plans with `stages` != 0 return NORM_ERR_PLAN, and with
 * a residual the fused add's 512-thread limit applies. */
norm_status ln_fwd_fp8_planned(const void* x, const void* residual, const void* gamma,
                               const void* beta, const float* scale, void* h, void* y8,
                               float* mean, float* rstd, int64_t M, int64_t N, float eps,
                               norm_dtype dtype, cudaStream_t stream, const norm_plan* plan);

norm_status rms_fwd_fp8_planned(const void* x, const void* residual, const void* w,
                                const float* scale, void* h, void* y8, int64_t M, int64_t N,
                                float eps, norm_dtype dtype, cudaStream_t stream,
                                const norm_plan* plan);

/* Static description of a status code. */
const char* norm_status_string(norm_status status);

/* cudaError_t of the last NORM_ERR_CUDA returned on the calling thread
 * (0 if none). */
int norm_last_cuda_error(void);

/* Version of this interface (bumped on any incompatible change). */
int norm_abi_version(void);

/*
 * Bounded waits. The only kernels that poll are the ring kernels (forward
 * plans with `stages` >= 2, and the backward plans norm_bwd_make_plan picks
 * for fp32 rows): a CTA waits for each bulk copy of an upcoming row on an
 * mbarrier, for at most the device's wait limit (2 s by default). When a
 * wait runs out, the whole CTA stops waiting and copying, gives the copies
 * it still has in flight one more wait of 2 s each (so that none lands in
 * the shared memory of a CTA that has gone), finishes and adds 1 to a count
 * on the device. The call's outputs are then void. Calls are asynchronous,
 * so they cannot return the timeout themselves: the caller asks afterwards.
 * The count and the limit belong to the current device; all calls on a
 * device share them. A cudaDeviceReset while the library is loaded is not
 * supported (the device address of that state is looked up once per device
 * and process).
 */

/* Reads the current device's count into *count and resets it to 0
 * (synchronises the device). NORM_ERR_ARG if count is NULL; NORM_ERR_CUDA on
 * a runtime error. */
norm_status norm_wait_timeouts(uint32_t* count);

/* Synchronises the current device and reports whether any ring wait ran out
 * since the last check: NORM_ERR_TIMEOUT if one did (and resets the count),
 * NORM_OK if none did, NORM_ERR_CUDA on a runtime error (for example one a
 * kernel raised). */
norm_status norm_synchronize(void);

/* Sets the current device's limit for the ring kernels' per-row waits, in
 * nanoseconds, for kernels launched after the call returns (synchronous;
 * call it while no ring kernel runs on the device). 0 makes every wait test
 * its copy once and give up if it has not landed yet (a way to exercise the
 * timeout path); the waits for copies in flight before a CTA exits keep
 * their own 2 s. NORM_ERR_ARG above 60 s (6e10 ns). */
norm_status norm_set_wait_limit(uint64_t ns);

/* The current device's per-row wait limit in nanoseconds (NORM_ERR_ARG if
 * ns is NULL). */
norm_status norm_wait_limit(uint64_t* ns);

#ifdef __cplusplus
}
#endif

#endif /* LIBNORM_H */
