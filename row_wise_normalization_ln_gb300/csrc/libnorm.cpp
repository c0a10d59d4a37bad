// libnorm C ABI: argument checks, the launch planner (which mapping, access
// width and register footprint a row gets) and dispatch to the kernels.
//
// Every argument error is caught here, before any CUDA call; nothing is
// launched on an error. The library allocates no memory and keeps no state
// between calls apart from a per-device cache of the SM count.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <initializer_list>

#include <cuda_runtime_api.h>

#include "libnorm.h"
#include "norm_args.h"

namespace {

using libnorm::NormArgs;

constexpr int64_t kMaxN = int64_t(1) << 24;  // fp32 counts are exact up to 2^24
constexpr int64_t kMaxGrid = int64_t(1) << 30;
constexpr int kMaxThreads = 1024;
constexpr int kMaxCluster = 8;               // portable cluster size
constexpr int kMaxPerThread = 8;
constexpr int64_t kMaxSmem = 225 * 1024;     // dynamic shared memory per CTA (below the 227 KB opt-in)
constexpr int kMaxStages = 4;

thread_local int g_last_cuda_error = 0;

bool dtype_ok(norm_dtype d) { return d == NORM_F32 || d == NORM_BF16 || d == NORM_F16; }
int elem_size(norm_dtype d) { return d == NORM_F32 ? 4 : 2; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }
int64_t pow2_ceil(int64_t v) {
    int64_t p = 1;
    while (p < v) p <<= 1;
    return p;
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// How the rows of a call can be accessed:
//   kAlignNone   element accesses only;
//   kAlignFull   every pointer 16-byte aligned and rows whole vectors: every
//                row starts on a 16-byte boundary;
//   kAlignPhase  the row tensors share their offset within 16 bytes (so
//                every row's elements sit at the same phase in each of
//                them): 16-byte vectors from each row's first aligned
//                element, the few elements around them one by one (CTA
//                mapping only).
enum AlignMode { kAlignNone = 0, kAlignFull = 1, kAlignPhase = 2 };

// The access mode of a call from its pointers: `rows` are the [M, N] row
// tensors (x, y and, when fused, the residual and h), `params` gamma/beta
// (or w); `y8` an FP8 output (one byte per element) or null.
int align_mode(std::initializer_list<const void*> rows, std::initializer_list<const void*> params, const void* y8,
               norm_dtype dtype, bool* vec_params) {
    const uintptr_t s = static_cast<uintptr_t>(elem_size(dtype));
    bool all16 = true, same = true;
    uintptr_t phase = 16;
    for (const void* p : rows) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        if (a % s != 0) return kAlignNone;  // not even element-aligned: element accesses
        if (phase == 16) phase = a & 15u;
        same = same && (a & 15u) == phase;
        all16 = all16 && (a & 15u) == 0;
    }
    bool pv = true;
    for (const void* p : params) pv = pv && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    *vec_params = pv;
    if (y8) {
        // the FP8 row's vector stores start where x's do: y8 and x/s agree modulo 16/s
        const uintptr_t vec = 16 / s;
        const uintptr_t x = reinterpret_cast<uintptr_t>(*rows.begin()) / s;
        if ((reinterpret_cast<uintptr_t>(y8) % vec) != (x % vec)) return kAlignNone;
        all16 = all16 && (reinterpret_cast<uintptr_t>(y8) & 15u) == 0;
    }
    if (!same) return kAlignNone;
    return (all16 && pv) ? kAlignFull : kAlignPhase;
}

// Checks shared by every entry point; M == 0 is legal.
norm_status check_sizes(int64_t M, int64_t N, norm_dtype dtype) {
    if (!dtype_ok(dtype)) return NORM_ERR_DTYPE;
    if (N < 1 || N > kMaxN || M < 0) return NORM_ERR_ARG;
    if (M > INT64_MAX / N) return NORM_ERR_ARG;
    return NORM_OK;
}


// Elements per access for this row shape and mode.
int vec_for(int64_t N, norm_dtype dtype, int mode) {
    const int s = elem_size(dtype);
    if (mode == kAlignFull && (N * s) % 16 == 0) return 16 / s;
    if (mode != kAlignNone) return 16 / s;  // phase-compatible rows (checked for the mapping by the caller)
    return 1;
}

// True when rows are whole 16-byte vectors on 16-byte boundaries.
bool rows_aligned(int64_t N, norm_dtype dtype, int mode) {
    return mode == kAlignFull && (N * elem_size(dtype)) % 16 == 0;
}

// The planner, from plan sweeps on GB300: rows do best with 8 accesses (128
// bytes) in registers per thread and CTAs of 64 to 256 threads; rows longer
// than 256 such threads go to a cluster of up to 8 CTAs of 128 threads, each
// walking its share in two rounds; lane groups only pay off below 64
// accesses per row.
norm_status make_plan(int64_t M, int64_t N, norm_dtype dtype, int mode, int num_sms, bool add, norm_plan* p) {
    std::memset(p, 0, sizeof *p);
    const int max_threads = add ? libnorm::kFusedMaxThreads : kMaxThreads;
    int vec = vec_for(N, dtype, mode);
    // Rows not on 16-byte boundaries take vectors only in the CTA mapping.
    if (vec > 1 && !rows_aligned(N, dtype, mode) && ceil_div(N, vec) < 64) vec = 1;
    const int64_t nacc = ceil_div(N, vec);
    const int64_t busy_threads = int64_t(num_sms) * 1024;  // half of the resident-thread capacity
    p->vec_elems = vec;

    // Short rows: a group of lanes per row, up to 8 accesses per lane.
    if (nacc < 64) {
        int64_t g = pow2_ceil(ceil_div(nacc, kMaxPerThread));
        if (g < 4) g = pow2_ceil(nacc < 4 ? nacc : 4);
        p->mapping = NORM_MAP_GROUP;
        p->group = static_cast<int32_t>(g);
        p->per_thread = static_cast<int32_t>(pow2_ceil(ceil_div(nacc, g)));
        p->threads = 256;
        p->cluster = 1;
        p->rounds = 1;
        p->grid = std::max<int64_t>(std::min<int64_t>(ceil_div(M, p->threads / g), kMaxGrid), 1);
        return NORM_OK;
    }

    // The fused residual add keeps two loads per access in flight: it runs
    // best with less per thread and more rounds (sweeps on GB300: LayerNorm
    // bf16 4096x8192 0.69 -> 0.82, fp32 2048x65536 0.72 -> 0.83 of the copy
    // bandwidth): 128-thread CTAs of 4 accesses per round, up to 4 rounds;
    // longer rows in clusters of up to 8 CTAs with 2 accesses per round.
    if (add) {
        int per = 4;
        int64_t threads = std::min<int64_t>(round_up(ceil_div(nacc, per), 32), 128);
        int64_t cluster = 1;
        if (ceil_div(nacc, threads * per) > 4) {
            per = 2;
            threads = 128;
            cluster = std::min<int64_t>(pow2_ceil(ceil_div(ceil_div(nacc, threads * per), 8)), kMaxCluster);
        }
        while (per > 1 && M * cluster * threads < busy_threads) {  // few rows: more threads
            const int64_t t2 = round_up(ceil_div(nacc, cluster * (per / 2)), 32);
            if (t2 > max_threads) break;
            per /= 2;
            threads = t2;
        }
        p->mapping = NORM_MAP_CTA;
        p->per_thread = per;
        p->threads = static_cast<int32_t>(threads);
        p->cluster = static_cast<int32_t>(cluster);
        p->rounds = static_cast<int32_t>(ceil_div(nacc, cluster * threads * per));
        p->grid = std::max<int64_t>(std::min<int64_t>(M, kMaxGrid / cluster), 1) * cluster;
        return NORM_OK;
    }

    // A CTA, or a cluster of CTAs, per row.
    int per = kMaxPerThread;
    int64_t threads = round_up(ceil_div(nacc, per), 32);
    if (threads < 64) {
        per = 4;
        threads = round_up(ceil_div(nacc, per), 32);
    }
    int64_t cluster = 1;
    if (threads > 256) {
        // Long rows: slices of 128 threads x 8 accesses, two register rounds
        // per slice, over a cluster of up to 8 CTAs (the second half of each
        // slice is read again from L2 for the output).
        const int64_t slices = ceil_div(nacc, int64_t(128) * per);
        cluster = std::min<int64_t>(pow2_ceil(ceil_div(slices, 2)), kMaxCluster);
        const int64_t rounds = ceil_div(slices, cluster);
        threads = std::min<int64_t>(round_up(ceil_div(nacc, cluster * per * rounds), 32), 128);
    }
    // Few rows: trade registers per thread for more threads per row.
    while (per > 1 && M * cluster * threads < busy_threads) {
        const int64_t t2 = round_up(ceil_div(nacc, cluster * (per / 2)), 32);
        if (t2 > max_threads) break;
        per /= 2;
        threads = t2;
    }
    if (threads < 32) threads = 32;
    p->mapping = NORM_MAP_CTA;
    p->per_thread = per;
    p->threads = static_cast<int32_t>(threads);
    p->cluster = static_cast<int32_t>(cluster);
    p->group = 0;
    p->rounds = static_cast<int32_t>(ceil_div(nacc, cluster * threads * per));
    p->grid = std::max<int64_t>(std::min<int64_t>(M, kMaxGrid / cluster), 1) * cluster;
    return NORM_OK;
}

// Validate an explicit plan against the call; derive `rounds`. The fused
// residual add (`add`) has no ring kernel and smaller CTAs.
norm_status check_plan(const norm_plan& in, int64_t N, norm_dtype dtype, int mode, bool add, bool q8,
                       norm_plan* out) {
    norm_plan p = in;
    if (add && (p.stages != 0 || p.threads > libnorm::kFusedMaxThreads)) return NORM_ERR_PLAN;
    if (q8 && p.stages != 0) return NORM_ERR_PLAN;
    const int s = elem_size(dtype);
    if (p.mapping != NORM_MAP_GROUP && p.mapping != NORM_MAP_CTA) return NORM_ERR_PLAN;
    if (p.vec_elems != 1) {
        if (p.vec_elems != 16 / s || mode == kAlignNone) return NORM_ERR_PLAN;
        // rows off 16-byte boundaries: the CTA register kernels only
        if (!rows_aligned(N, dtype, mode) && (p.mapping != NORM_MAP_CTA || p.stages != 0)) return NORM_ERR_PLAN;
    }
    if (!is_pow2(p.per_thread) || p.per_thread > kMaxPerThread) return NORM_ERR_PLAN;
    if (p.threads < 32 || p.threads > kMaxThreads || p.threads % 32 != 0) return NORM_ERR_PLAN;
    const int64_t nacc = ceil_div(N, p.vec_elems);
    if (p.mapping == NORM_MAP_GROUP) {
        if (!is_pow2(p.group) || p.group > 32) return NORM_ERR_PLAN;
        if (int64_t(p.group) * p.per_thread < nacc) return NORM_ERR_PLAN;
        if (p.stages != 0) return NORM_ERR_PLAN;
        p.cluster = 1;
        p.rounds = 1;
    } else {
        if (!is_pow2(p.cluster) || p.cluster > kMaxCluster) return NORM_ERR_PLAN;
        p.group = 0;
        p.rounds = static_cast<int32_t>(ceil_div(nacc, int64_t(p.cluster) * p.threads * p.per_thread));
    }
    if (p.stages != 0) {
        if (p.stages < 2 || p.stages > kMaxStages || p.vec_elems == 1 || p.rounds != 1) return NORM_ERR_PLAN;
        if (p.threads > libnorm::kRingMaxThreads) return NORM_ERR_PLAN;
        if (libnorm::ring_smem_bytes(p.stages, p.per_thread, p.threads) > kMaxSmem) return NORM_ERR_PLAN;
        if (p.grid == 0) {  // resolved at launch
            *out = p;
            return NORM_OK;
        }
    }
    if (p.grid < p.cluster || p.grid > kMaxGrid || p.grid % p.cluster != 0) return NORM_ERR_PLAN;
    *out = p;
    return NORM_OK;
}

// ------------------------------------------------------------ backward plans
// A backward plan covers a row in one register round: `cluster` CTAs of
// `threads` threads with `per_thread` accesses each. `group` is the launched
// cluster size: equal to `cluster` when a row spans several CTAs; otherwise
// the number of CTAs (each on its own rows) whose column accumulators are
// added through distributed shared memory before one partial row is
// written. `grid` is an upper bound on the CTAs launched (the launch takes
// no more than fit on the device at once); the workspace holds grid / group
// partial rows.
constexpr int kBwdMaxThreads = libnorm::kBwdMaxThreads;

int bwd_vmax(bool ln, norm_dtype dtype, int vec) {
    return vec == 1 ? 8 : (ln && elem_size(dtype) == 2) ? 2 : 4;
}

norm_status bwd_make_plan(int64_t M, int64_t N, norm_dtype dtype, bool all_aligned, int num_sms, bool ln,
                          norm_plan* p) {
    std::memset(p, 0, sizeof *p);
    const int vec = (all_aligned && (N * elem_size(dtype)) % 16 == 0) ? 16 / elem_size(dtype) : 1;
    const int64_t nacc = ceil_div(N, vec);
    int per = bwd_vmax(ln, dtype, vec);
    if (vec > 1) {
        // Vector rows: the fewest accesses per thread, from 2, that let one
        // CTA of at most 512 threads cover the row (sweeps on GB300: RMSNorm
        // fp32 8192x4096 72.1 -> 64.3 us with 512 x 2 instead of 256 x 4,
        // RMSNorm bf16 65536x2048 161 -> 127 us with 128 x 2 instead of
        // 64 x 4; one access per thread was slower).
        for (int q = std::min(2, per); q <= per; q *= 2)
            if (round_up(ceil_div(nacc, q), 32) <= kBwdMaxThreads) {
                per = q;
                break;
            }
    }
    int64_t cluster = 1;
    int64_t threads = round_up(ceil_div(nacc, per), 32);
    while (threads > kBwdMaxThreads && cluster < kMaxCluster) {
        cluster *= 2;
        threads = round_up(ceil_div(nacc, cluster * per), 32);
    }
    if (threads > kBwdMaxThreads) return NORM_ERR_ARG;  // the row does not fit one round of a cluster
    while (per > 1 && threads < 64) {
        per /= 2;
        threads = round_up(ceil_div(nacc, cluster * per), 32);
    }
    p->mapping = NORM_MAP_CTA;
    p->vec_elems = vec;
    p->per_thread = per;
    p->threads = static_cast<int32_t>(threads);
    p->cluster = static_cast<int32_t>(cluster);
    p->rounds = 1;
    // fp32 vector rows take a 2-stage ring of upcoming rows in shared memory
    // (measured on GB300: 10-15 % faster at 8192x4096, 8192x5000 and
    // 2048x65536; 3 or 4 stages slower); 16-bit vector rows of one CTA take
    // the register pipeline (LayerNorm bf16 4096x8192 54.6 -> 42.6 us,
    // RMSNorm bf16 65536x2048 146 -> 127 us).
    if (vec == 4 && libnorm::bwd_smem_bytes(ln, p->threads, per, vec, 2) <= kMaxSmem)
        p->stages = 2;
    else if (vec > 1 && cluster == 1)
        p->stages = 1;
    // Persistent grid of at most 1024 threads and 6 CTAs per SM in whole
    // clusters (the launch takes fewer if fewer fit at once). CTAs that each
    // take their own rows write one partial row each (no reduction cluster):
    // every SM takes part, and the column sum spreads the partial rows over
    // 32 warps per CTA (measured on GB300 against reduction clusters of 4
    // and 2: LayerNorm bf16 4096x8192 38.0 us against 40.7 and 38.8, RMSNorm
    // bf16 65536x2048 125.7 against 127.1, RMSNorm fp32 8192x4096 64.2
    // against 64.7 at 2).
    const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(6, 1024 / threads));
    if (cluster > 1) {
        const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(M, num_sms * per_sm / cluster));
        p->group = static_cast<int32_t>(cluster);
        p->grid = M > 0 ? clusters * cluster : 0;
    } else {
        const int64_t ctas = std::min<int64_t>(M, num_sms * per_sm);
        p->group = 1;
        p->grid = M > 0 ? ctas : 0;
    }
    return NORM_OK;
}

norm_status bwd_check_plan(const norm_plan& in, int64_t M, int64_t N, norm_dtype dtype, bool all_aligned, bool ln,
                           norm_plan* out) {
    norm_plan p = in;
    const int s = elem_size(dtype);
    if (p.mapping != NORM_MAP_CTA) return NORM_ERR_PLAN;
    if (p.vec_elems != 1) {
        if (p.vec_elems != 16 / s || !all_aligned || (N * s) % 16 != 0) return NORM_ERR_PLAN;
    }
    // stages 1: the register pipeline (a CTA per row); 2..4: the ring of
    // upcoming rows in shared memory (vector rows)
    if (p.stages == 1 && p.cluster != 1) return NORM_ERR_PLAN;
    if (p.stages != 0 && p.stages != 1 && (p.stages < 2 || p.stages > kMaxStages || p.vec_elems == 1))
        return NORM_ERR_PLAN;
    if (libnorm::bwd_smem_bytes(ln, p.threads, p.per_thread, p.vec_elems, p.stages) > kMaxSmem) return NORM_ERR_PLAN;
    if (!is_pow2(p.per_thread) || p.per_thread > bwd_vmax(ln, dtype, p.vec_elems)) return NORM_ERR_PLAN;
    if (p.threads < 32 || p.threads > kBwdMaxThreads || p.threads % 32 != 0) return NORM_ERR_PLAN;
    if (!is_pow2(p.cluster) || p.cluster > kMaxCluster) return NORM_ERR_PLAN;
    if (!is_pow2(p.group) || p.group > kMaxCluster) return NORM_ERR_PLAN;
    if (p.cluster > 1 && p.group != p.cluster) return NORM_ERR_PLAN;
    const int64_t nacc = ceil_div(N, p.vec_elems);
    if (int64_t(p.cluster) * p.threads * p.per_thread < nacc) return NORM_ERR_PLAN;  // one round only
    if (M > 0 && (p.grid < p.group || p.grid > kMaxGrid || p.grid % p.group != 0)) return NORM_ERR_PLAN;
    p.rounds = 1;
    if (M == 0) p.grid = 0;
    *out = p;
    return NORM_OK;
}

size_t bwd_workspace(const norm_plan& p, int64_t N, bool ln) {
    return static_cast<size_t>(libnorm::bwd_partials(p)) * (ln ? 2 : 1) * static_cast<size_t>(N) * sizeof(float);
}

// SM count of the current device (cached per device); `dev` receives the
// device ordinal.
int device_sm_count(int* dev_out) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        return -1;
    }
    *dev_out = dev;
    if (dev >= 0 && dev < 64) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || n <= 0) {
        g_last_cuda_error = static_cast<int>(e);
        return -1;
    }
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

using Launcher = cudaError_t (*)(const norm_plan&, const NormArgs&, cudaStream_t, int, int);

Launcher pick_launcher(bool ln, bool add, bool q8, norm_dtype dtype) {
    using namespace libnorm;
    // [q8][add][ln][dtype]
    static const Launcher table[2][2][2][3] = {
        {{{launch_rms_f32, launch_rms_bf16, launch_rms_f16}, {launch_ln_f32, launch_ln_bf16, launch_ln_f16}},
         {{launch_rms_add_f32, launch_rms_add_bf16, launch_rms_add_f16},
          {launch_ln_add_f32, launch_ln_add_bf16, launch_ln_add_f16}}},
        {{{launch_rms_fp8_f32, launch_rms_fp8_bf16, launch_rms_fp8_f16},
          {launch_ln_fp8_f32, launch_ln_fp8_bf16, launch_ln_fp8_f16}},
         {{launch_rms_add_fp8_f32, launch_rms_add_fp8_bf16, launch_rms_add_fp8_f16},
          {launch_ln_add_fp8_f32, launch_ln_add_fp8_bf16, launch_ln_add_fp8_f16}}}};
    return table[q8][add][ln][dtype];
}

// a.res != null selects the fused residual add; a.qscale != null the FP8
// output.
norm_status run(bool ln, const NormArgs& a, norm_dtype dtype, int mode, cudaStream_t stream,
                const norm_plan* user_plan) {
    const bool add = a.res != nullptr;
    const bool q8 = a.qscale != nullptr;
    norm_plan plan;
    if (user_plan) {
        const norm_status st = check_plan(*user_plan, a.N, dtype, mode, add, q8, &plan);
        if (st != NORM_OK) return st;
    }
    int dev = 0;
    const int sms = device_sm_count(&dev);
    if (sms <= 0) return NORM_ERR_CUDA;
    if (!user_plan) make_plan(a.M, a.N, dtype, mode, sms, add, &plan);
    NormArgs args = a;
    if (args.ldx == 0) args.ldx = a.N;  // contiguous rows
    if (args.ldy == 0) args.ldy = a.N;
    args.group = plan.group;
    args.rounds = plan.rounds;
    args.stages = plan.stages;
    args.shift = plan.vec_elems > 1 && !rows_aligned(a.N, dtype, mode);
    const cudaError_t e = pick_launcher(ln, add, q8, dtype)(plan, args, stream, sms, dev);
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        return NORM_ERR_CUDA;
    }
    return NORM_OK;
}

norm_status ln_impl(const void* x, const void* gamma, const void* beta, void* y, float* mean, float* rstd,
                    int64_t M, int64_t N, float eps, norm_dtype dtype, cudaStream_t stream, const norm_plan* plan) {
    norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return NORM_ERR_ARG;
    if (M == 0) return NORM_OK;
    if (!x || !gamma || !beta || !y) return NORM_ERR_ARG;
    bool vp = true;
    const int mode = align_mode({x, y}, {gamma, beta}, nullptr, dtype, &vp);
    NormArgs a{x, gamma, beta, y, mean, rstd, nullptr, nullptr, nullptr, M, static_cast<int32_t>(N), eps, 0, 1, 0};
    a.vec_params = vp;
    return run(true, a, dtype, mode, stream, plan);
}

norm_status rms_impl(const void* x, const void* w, void* y, int64_t M, int64_t N, float eps, norm_dtype dtype,
                     cudaStream_t stream, const norm_plan* plan) {
    norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return NORM_ERR_ARG;
    if (M == 0) return NORM_OK;
    if (!x || !w || !y) return NORM_ERR_ARG;
    bool vp = true;
    const int mode = align_mode({x, y}, {w}, nullptr, dtype, &vp);
    NormArgs a{x, w, nullptr, y, nullptr, nullptr, nullptr, nullptr, nullptr, M, static_cast<int32_t>(N), eps, 0, 1, 0};
    a.vec_params = vp;
    return run(false, a, dtype, mode, stream, plan);
}

// Fused residual add: h and y are both written, so they may not be the same
// buffer; each may be x or the residual itself.
norm_status ln_add_impl(const void* x, const void* res, const void* gamma, const void* beta, void* h, void* y,
                        float* mean, float* rstd, int64_t M, int64_t N, float eps, norm_dtype dtype,
                        cudaStream_t stream, const norm_plan* plan) {
    norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return NORM_ERR_ARG;
    if (M == 0) return NORM_OK;
    if (!x || !res || !gamma || !beta || !h || !y || h == y) return NORM_ERR_ARG;
    bool vp = true;
    const int mode = align_mode({x, res, h, y}, {gamma, beta}, nullptr, dtype, &vp);
    NormArgs a{x, gamma, beta, y, mean, rstd, res, h, nullptr, M, static_cast<int32_t>(N), eps, 0, 1, 0};
    a.vec_params = vp;
    return run(true, a, dtype, mode, stream, plan);
}

norm_status rms_add_impl(const void* x, const void* res, const void* w, void* h, void* y, int64_t M, int64_t N,
                         float eps, norm_dtype dtype, cudaStream_t stream, const norm_plan* plan) {
    norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return NORM_ERR_ARG;
    if (M == 0) return NORM_OK;
    if (!x || !res || !w || !h || !y || h == y) return NORM_ERR_ARG;
    bool vp = true;
    const int mode = align_mode({x, res, h, y}, {w}, nullptr, dtype, &vp);
    NormArgs a{x, w, nullptr, y, nullptr, nullptr, res, h, nullptr, M, static_cast<int32_t>(N), eps, 0, 1, 0};
    a.vec_params = vp;
    return run(false, a, dtype, mode, stream, plan);
}

// Strided rows: x and y rows ldx and ldy elements apart (>= N). The access
// mode then also looks at the pitches: full vectors need pitches of whole
// 16-byte vectors, a shared phase needs the pitches to agree modulo 16 bytes.
norm_status strided_impl(bool ln, const void* x, int64_t ldx, const void* gamma, const void* beta, void* y,
                         int64_t ldy, float* mean, float* rstd, int64_t M, int64_t N, float eps, norm_dtype dtype,
                         cudaStream_t stream, const norm_plan* plan) {
    norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return NORM_ERR_ARG;
    if (ldx < N || ldy < N) return NORM_ERR_ARG;
    if (M == 0) return NORM_OK;
    if ((M - 1) > (INT64_MAX - N) / std::max(ldx, ldy)) return NORM_ERR_ARG;
    if (!x || !gamma || (ln && !beta) || !y) return NORM_ERR_ARG;
    const int64_t s = elem_size(dtype);
    bool vp = true;
    int mode = ln ? align_mode({x, y}, {gamma, beta}, nullptr, dtype, &vp) : align_mode({x, y}, {gamma}, nullptr, dtype, &vp);
    if (mode != kAlignNone && ((ldx * s) & 15) != ((ldy * s) & 15)) mode = kAlignNone;
    if (mode == kAlignFull && ((ldx * s) & 15) != 0) mode = kAlignPhase;
    NormArgs a{x, gamma, ln ? beta : nullptr, y, ln ? mean : nullptr, ln ? rstd : nullptr, nullptr, nullptr, nullptr,
               M, static_cast<int32_t>(N), eps, 0, 1, 0};
    a.ldx = ldx;
    a.ldy = ldy;
    a.vec_params = vp;
    return run(ln, a, dtype, mode, stream, plan);
}

// FP8 output: y8 holds one E4M3 byte per element; scale is one fp32 value
// in device memory. With a residual (res != null) also h = x + res.
norm_status fp8_impl(bool ln, const void* x, const void* res, const void* gamma, const void* beta,
                     const float* scale, void* h, void* y8, float* mean, float* rstd, int64_t M, int64_t N,
                     float eps, norm_dtype dtype, cudaStream_t stream, const norm_plan* plan) {
    norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return NORM_ERR_ARG;
    if (M == 0) return NORM_OK;
    if (!x || !gamma || (ln && !beta) || !scale || !y8) return NORM_ERR_ARG;
    if (res && (!h || h == y8)) return NORM_ERR_ARG;
    bool vp = true;
    const int mode = res ? align_mode({x, res, h}, {gamma, ln ? beta : gamma}, y8, dtype, &vp)
                         : align_mode({x}, {gamma, ln ? beta : gamma}, y8, dtype, &vp);
    NormArgs a{x, gamma, ln ? beta : nullptr, y8, ln ? mean : nullptr, ln ? rstd : nullptr, res, res ? h : nullptr,
               scale, M, static_cast<int32_t>(N), eps, 0, 1, 0};
    a.vec_params = vp;
    return run(ln, a, dtype, mode, stream, plan);
}

// Backward: dx = d(loss)/dx for y = norm(x); column gradients in fp32.
norm_status bwd_impl(bool ln, const void* dy, const void* x, const void* gamma, const float* mean, const float* rstd,
                     void* dx, float* dgamma, float* dbeta, void* ws, size_t ws_bytes, int64_t M, int64_t N,
                     float eps, norm_dtype dtype, cudaStream_t stream, const norm_plan* user_plan) {
    norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!std::isfinite(eps) || eps < 0.f) return NORM_ERR_ARG;
    if (!dgamma || (ln && !dbeta)) return NORM_ERR_ARG;
    if (M > 0 && (!dy || !x || !gamma || !dx || (ln && (!mean || !rstd)))) return NORM_ERR_ARG;
    const bool al = aligned16(dy) && aligned16(x) && aligned16(gamma) && aligned16(dx);
    {
        norm_plan probe;  // rows beyond the backward's limit fail here, before any CUDA call
        st = bwd_make_plan(M, N, dtype, al, 1, ln, &probe);
        if (st != NORM_OK) return st;
    }
    auto ws_ok = [&](const norm_plan& pl) {
        const size_t need = bwd_workspace(pl, N, ln);
        return need == 0 || (ws && ws_bytes >= need && (reinterpret_cast<uintptr_t>(ws) & 15u) == 0);
    };
    norm_plan plan;
    if (user_plan) {
        st = bwd_check_plan(*user_plan, M, N, dtype, al, ln, &plan);
        if (st != NORM_OK) return st;
        if (!ws_ok(plan)) return NORM_ERR_ARG;
    }
    int dev = 0;
    const int sms = device_sm_count(&dev);
    if (sms <= 0) return NORM_ERR_CUDA;
    if (!user_plan) {
        st = bwd_make_plan(M, N, dtype, al, sms, ln, &plan);
        if (st != NORM_OK) return st;
        if (!ws_ok(plan)) return NORM_ERR_ARG;
    }
    libnorm::BwdArgs a{dy, x, gamma, mean, rstd, dx, static_cast<float*>(ws), dgamma, dbeta, M,
                       static_cast<int32_t>(N), eps, plan.cluster};
    using BwdLauncher = cudaError_t (*)(const norm_plan&, const libnorm::BwdArgs&, cudaStream_t, int, int);
    static const BwdLauncher table[2][3] = {
        {libnorm::launch_rms_bwd_f32, libnorm::launch_rms_bwd_bf16, libnorm::launch_rms_bwd_f16},
        {libnorm::launch_ln_bwd_f32, libnorm::launch_ln_bwd_bf16, libnorm::launch_ln_bwd_f16}};
    const cudaError_t e = table[ln][dtype](plan, a, stream, dev, sms);
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        return NORM_ERR_CUDA;
    }
    return NORM_OK;
}

}  // namespace

void libnorm::note_cuda_error(int e) { g_last_cuda_error = e; }

extern "C" {

norm_status ln_bwd(const void* dy, const void* x, const void* gamma, const float* mean, const float* rstd, void* dx,
                   float* dgamma, float* dbeta, void* workspace, size_t workspace_bytes, int64_t M, int64_t N,
                   norm_dtype dtype, cudaStream_t stream) {
    return bwd_impl(true, dy, x, gamma, mean, rstd, dx, dgamma, dbeta, workspace, workspace_bytes, M, N, 0.f, dtype,
                    stream, nullptr);
}

norm_status rms_bwd(const void* dy, const void* x, const void* w, void* dx, float* dw, void* workspace,
                    size_t workspace_bytes, int64_t M, int64_t N, float eps, norm_dtype dtype, cudaStream_t stream) {
    return bwd_impl(false, dy, x, w, nullptr, nullptr, dx, dw, nullptr, workspace, workspace_bytes, M, N, eps, dtype,
                    stream, nullptr);
}

norm_status ln_bwd_planned(const void* dy, const void* x, const void* gamma, const float* mean, const float* rstd,
                           void* dx, float* dgamma, float* dbeta, void* workspace, size_t workspace_bytes, int64_t M,
                           int64_t N, norm_dtype dtype, cudaStream_t stream, const norm_plan* plan) {
    return bwd_impl(true, dy, x, gamma, mean, rstd, dx, dgamma, dbeta, workspace, workspace_bytes, M, N, 0.f, dtype,
                    stream, plan);
}

norm_status rms_bwd_planned(const void* dy, const void* x, const void* w, void* dx, float* dw, void* workspace,
                            size_t workspace_bytes, int64_t M, int64_t N, float eps, norm_dtype dtype,
                            cudaStream_t stream, const norm_plan* plan) {
    return bwd_impl(false, dy, x, w, nullptr, nullptr, dx, dw, nullptr, workspace, workspace_bytes, M, N, eps, dtype,
                    stream, plan);
}

norm_status norm_bwd_make_plan(int64_t M, int64_t N, norm_dtype dtype, int layer_norm, int aligned, int num_sms,
                               norm_plan* plan) {
    const norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!plan || num_sms < 1) return NORM_ERR_ARG;
    return bwd_make_plan(M, N, dtype, aligned != 0, num_sms, layer_norm != 0, plan);
}

norm_status norm_bwd_workspace_bytes(const norm_plan* plan, int64_t N, int layer_norm, size_t* bytes) {
    if (!plan || !bytes || N < 1 || N > kMaxN || plan->group < 1 || plan->grid < 0) return NORM_ERR_ARG;
    *bytes = bwd_workspace(*plan, N, layer_norm != 0);
    return NORM_OK;
}

norm_status ln_fwd(const void* x, const void* gamma, const void* beta, void* y, float* mean, float* rstd,
                   int64_t M, int64_t N, float eps, norm_dtype dtype, cudaStream_t stream) {
    return ln_impl(x, gamma, beta, y, mean, rstd, M, N, eps, dtype, stream, nullptr);
}

norm_status rms_fwd(const void* x, const void* w, void* y, int64_t M, int64_t N, float eps, norm_dtype dtype,
                    cudaStream_t stream) {
    return rms_impl(x, w, y, M, N, eps, dtype, stream, nullptr);
}

norm_status ln_fwd_planned(const void* x, const void* gamma, const void* beta, void* y, float* mean, float* rstd,
                           int64_t M, int64_t N, float eps, norm_dtype dtype, cudaStream_t stream,
                           const norm_plan* plan) {
    return ln_impl(x, gamma, beta, y, mean, rstd, M, N, eps, dtype, stream, plan);
}

norm_status rms_fwd_planned(const void* x, const void* w, void* y, int64_t M, int64_t N, float eps,
                            norm_dtype dtype, cudaStream_t stream, const norm_plan* plan) {
    return rms_impl(x, w, y, M, N, eps, dtype, stream, plan);
}

norm_status ln_fwd_add(const void* x, const void* residual, const void* gamma, const void* beta, void* h, void* y,
                       float* mean, float* rstd, int64_t M, int64_t N, float eps, norm_dtype dtype,
                       cudaStream_t stream) {
    return ln_add_impl(x, residual, gamma, beta, h, y, mean, rstd, M, N, eps, dtype, stream, nullptr);
}

norm_status rms_fwd_add(const void* x, const void* residual, const void* w, void* h, void* y, int64_t M, int64_t N,
                        float eps, norm_dtype dtype, cudaStream_t stream) {
    return rms_add_impl(x, residual, w, h, y, M, N, eps, dtype, stream, nullptr);
}

norm_status ln_fwd_add_planned(const void* x, const void* residual, const void* gamma, const void* beta, void* h,
                               void* y, float* mean, float* rstd, int64_t M, int64_t N, float eps,
                               norm_dtype dtype, cudaStream_t stream, const norm_plan* plan) {
    return ln_add_impl(x, residual, gamma, beta, h, y, mean, rstd, M, N, eps, dtype, stream, plan);
}

norm_status rms_fwd_add_planned(const void* x, const void* residual, const void* w, void* h, void* y, int64_t M,
                                int64_t N, float eps, norm_dtype dtype, cudaStream_t stream,
                                const norm_plan* plan) {
    return rms_add_impl(x, residual, w, h, y, M, N, eps, dtype, stream, plan);
}

norm_status ln_fwd_strided(const void* x, int64_t ldx, const void* gamma, const void* beta, void* y, int64_t ldy,
                           float* mean, float* rstd, int64_t M, int64_t N, float eps, norm_dtype dtype,
                           cudaStream_t stream, const norm_plan* plan) {
    return strided_impl(true, x, ldx, gamma, beta, y, ldy, mean, rstd, M, N, eps, dtype, stream, plan);
}

norm_status rms_fwd_strided(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy, int64_t M, int64_t N,
                            float eps, norm_dtype dtype, cudaStream_t stream, const norm_plan* plan) {
    return strided_impl(false, x, ldx, w, nullptr, y, ldy, nullptr, nullptr, M, N, eps, dtype, stream, plan);
}

norm_status ln_fwd_fp8(const void* x, const void* gamma, const void* beta, const float* scale, void* y8, float* mean,
                       float* rstd, int64_t M, int64_t N, float eps, norm_dtype dtype, cudaStream_t stream) {
    return fp8_impl(true, x, nullptr, gamma, beta, scale, nullptr, y8, mean, rstd, M, N, eps, dtype, stream, nullptr);
}

norm_status rms_fwd_fp8(const void* x, const void* w, const float* scale, void* y8, int64_t M, int64_t N, float eps,
                        norm_dtype dtype, cudaStream_t stream) {
    return fp8_impl(false, x, nullptr, w, nullptr, scale, nullptr, y8, nullptr, nullptr, M, N, eps, dtype, stream,
                    nullptr);
}

norm_status ln_fwd_add_fp8(const void* x, const void* residual, const void* gamma, const void* beta,
                           const float* scale, void* h, void* y8, float* mean, float* rstd, int64_t M, int64_t N,
                           float eps, norm_dtype dtype, cudaStream_t stream) {
    if (!residual) return NORM_ERR_ARG;
    return fp8_impl(true, x, residual, gamma, beta, scale, h, y8, mean, rstd, M, N, eps, dtype, stream, nullptr);
}

norm_status rms_fwd_add_fp8(const void* x, const void* residual, const void* w, const float* scale, void* h,
                            void* y8, int64_t M, int64_t N, float eps, norm_dtype dtype, cudaStream_t stream) {
    if (!residual) return NORM_ERR_ARG;
    return fp8_impl(false, x, residual, w, nullptr, scale, h, y8, nullptr, nullptr, M, N, eps, dtype, stream,
                    nullptr);
}

norm_status ln_fwd_fp8_planned(const void* x, const void* residual, const void* gamma, const void* beta,
                               const float* scale, void* h, void* y8, float* mean, float* rstd, int64_t M, int64_t N,
                               float eps, norm_dtype dtype, cudaStream_t stream, const norm_plan* plan) {
    return fp8_impl(true, x, residual, gamma, beta, scale, h, y8, mean, rstd, M, N, eps, dtype, stream, plan);
}

norm_status rms_fwd_fp8_planned(const void* x, const void* residual, const void* w, const float* scale, void* h,
                                void* y8, int64_t M, int64_t N, float eps, norm_dtype dtype, cudaStream_t stream,
                                const norm_plan* plan) {
    return fp8_impl(false, x, residual, w, nullptr, scale, h, y8, nullptr, nullptr, M, N, eps, dtype, stream, plan);
}

norm_status norm_make_plan(int64_t M, int64_t N, norm_dtype dtype, int aligned, int num_sms, norm_plan* plan) {
    const norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!plan || num_sms < 1) return NORM_ERR_ARG;
    if (aligned < kAlignNone || aligned > kAlignPhase) return NORM_ERR_ARG;
    return make_plan(M, N, dtype, aligned, num_sms, false, plan);
}

norm_status norm_make_plan_add(int64_t M, int64_t N, norm_dtype dtype, int aligned, int num_sms, norm_plan* plan) {
    const norm_status st = check_sizes(M, N, dtype);
    if (st != NORM_OK) return st;
    if (!plan || num_sms < 1) return NORM_ERR_ARG;
    if (aligned < kAlignNone || aligned > kAlignPhase) return NORM_ERR_ARG;
    return make_plan(M, N, dtype, aligned, num_sms, true, plan);
}

const char* norm_status_string(norm_status s) {
    switch (s) {
        case NORM_OK: return "ok";
        case NORM_ERR_ARG: return "invalid argument (size, pointer or eps)";
        case NORM_ERR_DTYPE: return "unsupported dtype";
        case NORM_ERR_CUDA: return "CUDA runtime error (see norm_last_cuda_error)";
        case NORM_ERR_PLAN: return "plan inconsistent with the call";
        case NORM_ERR_TIMEOUT: return "a ring kernel's wait for a bulk copy ran out (outputs void)";
        default: return "unknown status";
    }
}

int norm_last_cuda_error(void) { return g_last_cuda_error; }

int norm_abi_version(void) { return 1; }

}  // extern "C"
