// Row-wise LayerNorm / RMSNorm backward kernels for sm_103a.
//
// LayerNorm ([Ch7] §7.7), per row with the forward's saved mean and rstd:
//     xhat = (x - mean) * rstd,   g = dy * gamma,
//     dx   = rstd * (g - mean_j(g) - xhat * mean_j(g * xhat)),
// and over rows dgamma = sum dy * xhat, dbeta = sum dy. The two row sums are
// reduced together as one pair (butterfly, shared memory, distributed shared
// memory across a cluster), as the chapter suggests.
// RMSNorm ([Ch7] §7.7, last paragraph): rstd is recomputed from the row in
// registers (the forward keeps no statistics), so the pair is
// (sum x^2, sum dy * w * x):
//     dx = rstd * w * dy - x * rstd^3 * sum(dy * w * x) / N,   dw = sum dy * x * rstd.
//
// norm_bwd_cta: a CTA, or a cluster of CTAs, owns one row at a time (one
// register round; x and dy are read once) and walks rows in a grid-stride
// loop, with the rows two steps ahead prefetched into L2. A thread owns the same columns in every row it visits, so it
// accumulates the column gradients of those columns in its own slots of
// shared memory. At the end, CTAs that share columns (the CTAs of a
// reduction cluster, each on its own rows) add their accumulators through
// distributed shared memory, and each cluster writes one partial row to the
// workspace.
// norm_bwd_colsum: sums the partial rows of every column in a fixed order,
// so the column gradients are deterministic for a given plan.
//
// Sources (page title, section): [Ch7] "第 7 章 LayerNorm 与 RMSNorm" §7.7;
// [T3] "T3 讲解：LayerNorm / RMSNorm 的 forward" §⑥ (mean and rstd are saved
// in fp32 for the backward).
#pragma once

#include <map>
#include <mutex>
#include <tuple>

#include "norm_kernels.cuh"

namespace libnorm {

// Element i (widened to fp32) of one access, and an access rounded from
// VEC fp32 values.
template <class T, int VEC>
struct BwdElem;

template <>
struct BwdElem<float, 4> {
    using Raw = uint4;
    static __device__ __forceinline__ float get(const Raw& r, int i) { return Ops<float, 4>::e(r, i); }
    static __device__ __forceinline__ Raw pack(const float* v) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
    }
};

template <class T, class P>
struct BwdElem16 {
    using Raw = uint4;
    static __device__ __forceinline__ float get(const Raw& r, int i) {
        const float2 f = P::widen(Ops16<T, P>::w(r, i >> 1));
        return (i & 1) ? f.y : f.x;
    }
    static __device__ __forceinline__ Raw pack(const float* v) {
        return make_uint4(P::pack(v[0], v[1]), P::pack(v[2], v[3]), P::pack(v[4], v[5]), P::pack(v[6], v[7]));
    }
};
template <>
struct BwdElem<__nv_bfloat16, 8> : BwdElem16<__nv_bfloat16, Bf16Pair> {};
template <>
struct BwdElem<__half, 8> : BwdElem16<__half, F16Pair> {};

// The pair codec of a 16-bit element type.
template <class T>
struct PairOf {
    using type = Bf16Pair;
};
template <>
struct PairOf<__half> {
    using type = F16Pair;
};

template <class T>
struct BwdElem<T, 1> {
    using Raw = uint32_t;
    static __device__ __forceinline__ float get(Raw r, int) { return ScalarOps<T>::e(r); }
    static __device__ __forceinline__ Raw pack(const float* v) { return ScalarOps<T>::from_float(v[0]); }
};

// ------------------------------------------------------------ pair reduction
// Sum of a pair of values per thread over the CTA and, when C > 1, over the
// cluster; every thread of every CTA of the cluster gets the same bits.
// Slots alternate by `stage` (the row's parity), so a slot is written again
// only after a barrier every reader of its previous value has passed.
struct PairReduceSmem {
    float2 warp_part[2][32];
    float2 cta_part[2];
};

__device__ __forceinline__ float2 ld_peer_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float2 row_sum2(PairReduceSmem& red, int stage, float2 v, int C, int nwarps,
                                           int wwidth) {
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    v.x = group_sum(v.x, 32);
    v.y = group_sum(v.y, 32);
    if (lane == 0) red.warp_part[stage][tid >> 5] = v;
    __syncthreads();
    float2 w = lane < nwarps ? red.warp_part[stage][lane] : make_float2(0.f, 0.f);
    w.x = sum_first_lanes(w.x, wwidth);
    w.y = sum_first_lanes(w.y, wwidth);
    if (C > 1) {
        if (tid == 0) red.cta_part[stage] = w;
        cluster_barrier();
        const float2 p =
            lane < C ? ld_peer_f32x2(peer_smem_addr(&red.cta_part[stage], static_cast<uint32_t>(lane)))
                     : make_float2(0.f, 0.f);
        w.x = sum_first_lanes(p.x, C);
        w.y = sum_first_lanes(p.y, C);
    }
    return w;
}

// ------------------------------------------------------------ main kernel
// Layout as the forward's CTA mapping: CTA rank k of a row's cluster holds
// accesses [k*V*T, (k+1)*V*T), warp-major. Launched as clusters of Q CTAs:
// Q == row_cluster when a row spans a cluster; with row_cluster == 1 the Q
// CTAs of a cluster each take their own rows and meet only at the end.
//
// Each thread keeps gamma (w) of its columns in registers for the whole
// kernel. Rows two steps ahead are prefetched into L2 (bulk, by one thread),
// so a row's own loads are L2 hits while HBM already serves the rows after
// it. (Loads into registers issued a row ahead did not overlap: the row's
// block barrier waits for them.) The column accumulators live in registers
// (in this thread's shared-memory slots for the 16-bit variants of 4
// accesses per thread); at the end they sit in dynamic shared memory,
// [NA][T*V*VEC] floats, each thread at the positions of its own columns.
template <class T, int VEC, int V, bool LN, bool RING>
__global__ void __launch_bounds__(kBwdMaxThreads) norm_bwd_cta(const BwdArgs a) {
    static_assert(!RING || VEC > 1, "the ring moves 16-byte vectors");
    using O = OpsFor<T, VEC>;
    using E = BwdElem<T, VEC>;
    using Raw = typename O::Raw;
    constexpr int NA = LN ? 2 : 1;
    __shared__ PairReduceSmem red;
    extern __shared__ float4 acc_v[];
    float* acc_s = reinterpret_cast<float*>(acc_v);

    const int T_ = blockDim.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T_ >> 5;
    int wwidth = 1;
    while (wwidth < nwarps) wwidth <<= 1;
    const uint32_t Q = cluster_size();
    const uint32_t crank = cluster_rank();
    const int C = a.row_cluster;
    const int rank = C > 1 ? static_cast<int>(crank) : 0;
    const int64_t first_row = C > 1 ? blockIdx.x / C : blockIdx.x;
    const int64_t row_step = C > 1 ? gridDim.x / C : gridDim.x;
    const int N = a.N;
    const int nacc = (N + VEC - 1) / VEC;
    const int stride = 32 * VEC;
    const int local = warp * V * 32 + lane;  // first access within this CTA's slice
    const int f0 = rank * V * T_ + local;    // ... within the row
    const int nv = valid_runs(nacc, f0, 32, V);
    const float invN = 1.f / static_cast<float>(N);
    const int slice = T_ * V * VEC;  // floats per accumulator array
    float* my_acc = acc_s + local * VEC;
    // RING: after the accumulators, `stages` stages of this CTA's slices of
    // an upcoming row, x then dy (V*T 16-byte slots each), then one mbarrier
    // per stage.
    const int stages = RING ? a.stages : 0;
    uint4* ring = reinterpret_cast<uint4*>(acc_s + NA * slice);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + 2 * stages * V * T_);

    // Column accumulators in registers where they fit beside the row data
    // (all but the 16-bit variants of 4 accesses per thread); otherwise in
    // this thread's shared-memory slots.
    constexpr bool ACC_REG = !(VEC == 8 && V >= 4);
    float acc[ACC_REG ? NA : 1][ACC_REG ? V : 1][ACC_REG ? VEC : 1];
#pragma unroll
    for (int k = 0; k < (ACC_REG ? NA : 1); ++k)
#pragma unroll
        for (int j = 0; j < (ACC_REG ? V : 1); ++j)
#pragma unroll
            for (int e = 0; e < (ACC_REG ? VEC : 1); ++e) acc[k][j][e] = 0.f;
    // Shared-memory accumulator slots start at zero.
#pragma unroll
    for (int k = 0; k < (ACC_REG ? 0 : NA); ++k)
#pragma unroll
        for (int j = 0; j < V; ++j)
#pragma unroll
            for (int e = 0; e < VEC; e += (VEC % 4 == 0 ? 4 : 1)) {
                float* d = my_acc + k * slice + j * 32 * VEC + e;
                if constexpr (VEC % 4 == 0)
                    *reinterpret_cast<float4*>(d) = make_float4(0.f, 0.f, 0.f, 0.f);
                else
                    *d = 0.f;
            }

    // Rows ahead go to L2 by bulk prefetch: this CTA's contiguous slice of x
    // and dy (16-byte vector rows only) and the row's statistics, issued by
    // one thread, two rows ahead of the row being worked on.
    const int64_t cta_first = static_cast<int64_t>(rank) * V * T_ * VEC;  // first element of the CTA's slice
    const uint32_t slice_bytes = static_cast<uint32_t>(
        (cta_first < N ? min(static_cast<int64_t>(V) * T_ * VEC, N - cta_first) : 0) * sizeof(T));
    auto prefetch_row = [&](int64_t r) {
        if (r >= a.M) return;
        if constexpr (VEC > 1) {
            if (slice_bytes > 0) {
                prefetch_l2_bulk(static_cast<const T*>(a.x) + r * N + cta_first, slice_bytes);
                prefetch_l2_bulk(static_cast<const T*>(a.dy) + r * N + cta_first, slice_bytes);
            }
        }
        if constexpr (LN) {
            prefetch_l2_line(a.mean + r);
            prefetch_l2_line(a.rstd + r);
        }
    };
    // Rows are prefetched `ahead` rows before their turn: 2 without a ring;
    // with one, one row beyond those in the ring, so that each bulk copy
    // into the ring reads L2. The first rows are requested before the
    // dependent-launch wait, overlapping the previous grid's tail (a
    // prefetch only moves data towards L2, where that grid's writes land).
    const int ahead = RING ? stages + 1 : 2;
    if (tid == 0)
        for (int k = 0; k < ahead; ++k) prefetch_row(first_row + k * row_step);
    if constexpr (RING) {
        if (tid == 0) {
            for (int k = 0; k < stages; ++k) mbar_init(&full[k], 1);
            mbar_init_fence();
        }
        __syncthreads();
    }

    grid_release();
    grid_wait();

    // RING, thread 0: fill stage `st` with this CTA's slices of x and dy of
    // row `r` (copies read memory: only after the wait above).
    auto issue = [&](int64_t r, int st) {
        mbar_arrive_expect(&full[st], 2u * slice_bytes);
        if (slice_bytes > 0) {
            bulk_load(ring + (2 * st) * V * T_, static_cast<const T*>(a.x) + r * N + cta_first, slice_bytes,
                      &full[st]);
            bulk_load(ring + (2 * st + 1) * V * T_, static_cast<const T*>(a.dy) + r * N + cta_first, slice_bytes,
                      &full[st]);
        }
    };
    if constexpr (RING) {
        if (tid == 0)
            for (int k = 0; k < stages; ++k)
                if (first_row + k * row_step < a.M) issue(first_row + k * row_step, k);
    }

    // 16-bit rows work on fp32 pairs with the packed instructions and keep
    // gamma widened (gf); other rows work on scalars.
    constexpr bool PAIRS = VEC == 8;
    using P = typename PairOf<T>::type;
    Raw gv[V];
    float2 gf[PAIRS ? V : 1][4];
    {
        const T* gp = static_cast<const T*>(a.gamma) + f0 * VEC;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nv) {
                gv[j] = O::load_param(gp + j * stride);
                if constexpr (PAIRS) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) gf[j][i] = P::widen(Ops16<T, P>::w(gv[j], i));
                }
            }
    }
    const T* xbase = static_cast<const T*>(a.x) + f0 * VEC;
    const T* dybase = static_cast<const T*>(a.dy) + f0 * VEC;

    int it = 0;
    int st = 0;            // RING: this row's stage
    uint32_t parity = 0;   // ... and the phase parity to wait for
    int64_t late = -1;     // RING: the row (count) whose wait ran out, if any
    for (int64_t row = first_row; row < a.M; row += row_step, ++it) {
        if (tid == 0) prefetch_row(row + ahead * row_step);
        Raw xv[V], dv[V];
        if constexpr (RING) {
            // After one wait has run out this CTA neither waits nor copies
            // any more (its outputs are void by then); the kernel still ends.
            if (late < 0 && !mbar_wait(&full[st], parity)) late = it;
            const uint4* xs = ring + (2 * st) * V * T_ + local;
            const uint4* ds = xs + V * T_;
#pragma unroll
            for (int j = 0; j < V; ++j)
                if (j < nv) {
                    xv[j] = xs[j * 32];
                    dv[j] = ds[j * 32];
                }
        } else {
#pragma unroll
            for (int j = 0; j < V; ++j)
                if (j < nv) {
                    xv[j] = O::load(xbase + row * N + j * stride);
                    dv[j] = O::load(dybase + row * N + j * stride);
                }
        }
        float mu = 0.f, rs = 0.f;
        if constexpr (LN) {
            mu = a.mean[row];
            rs = a.rstd[row];
        }
        float s0 = 0.f, s1 = 0.f;
        if constexpr (PAIRS) {
            const float2 nmu = f2_splat(-mu), rs2 = f2_splat(rs);
            float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < V; ++j)
                if (j < nv) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 x2 = P::widen(Ops16<T, P>::w(xv[j], i));
                        const float2 d2 = P::widen(Ops16<T, P>::w(dv[j], i));
                        if constexpr (LN) {
                            const float2 xh = __fmul2_rn(__fadd2_rn(x2, nmu), rs2);
                            const float2 g = __fmul2_rn(d2, gf[j][i]);
                            a0 = __fadd2_rn(a0, g);
                            a1 = __ffma2_rn(g, xh, a1);
                        } else {
                            a0 = __ffma2_rn(x2, x2, a0);
                            a1 = __ffma2_rn(__fmul2_rn(d2, gf[j][i]), x2, a1);
                        }
                    }
                }
            s0 = a0.x + a0.y;
            s1 = a1.x + a1.y;
        } else {
#pragma unroll
            for (int j = 0; j < V; ++j)
                if (j < nv) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float xe = E::get(xv[j], e), de = E::get(dv[j], e), ge = E::get(gv[j], e);
                        if constexpr (LN) {
                            const float xh = (xe - mu) * rs;
                            const float g = de * ge;
                            s0 += g;
                            s1 = fmaf(g, xh, s1);
                        } else {
                            s0 = fmaf(xe, xe, s0);
                            s1 = fmaf(de * ge, xe, s1);
                        }
                    }
                }
        }
        const float2 S = row_sum2(red, it & 1, make_float2(s0, s1), C, nwarps, wwidth);
        if constexpr (RING) {
            // Every thread has read this stage before the barrier above:
            // refill it with the row `stages` turns ahead.
            if (tid == 0 && late < 0 && row + stages * row_step < a.M) {
                fence_proxy_async();
                issue(row + stages * row_step, st);
            }
            if (++st == stages) st = 0, parity ^= 1u;
        }
        T* dxr = static_cast<T*>(a.dx) + row * N + f0 * VEC;
        float c0, c1;  // LayerNorm: mean(g), mean(g xhat); RMSNorm: rstd, rstd^3 mean(dy w x)
        if constexpr (LN) {
            c0 = S.x * invN;
            c1 = S.y * invN;
        } else {
            c0 = rsqrtf(S.x * invN + a.eps);
            c1 = c0 * c0 * c0 * (S.y * invN);
        }
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nv) {
                float o[VEC], pa[VEC], pb[VEC];
                if constexpr (PAIRS) {
                    const float2 nmu = f2_splat(-mu), rs2 = f2_splat(rs), nc0 = f2_splat(-c0), nc1 = f2_splat(-c1),
                                 c02 = f2_splat(c0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 x2 = P::widen(Ops16<T, P>::w(xv[j], i));
                        const float2 d2 = P::widen(Ops16<T, P>::w(dv[j], i));
                        float2 ov, av = make_float2(0.f, 0.f), bv = d2;
                        if constexpr (LN) {
                            const float2 xh = __fmul2_rn(__fadd2_rn(x2, nmu), rs2);
                            const float2 t = __fadd2_rn(__fmul2_rn(d2, gf[j][i]), nc0);
                            ov = __fmul2_rn(rs2, __ffma2_rn(xh, nc1, t));
                            if constexpr (ACC_REG) {
                                const float2 ga = __ffma2_rn(d2, xh, make_float2(acc[0][j][2 * i], acc[0][j][2 * i + 1]));
                                const float2 gb = __fadd2_rn(make_float2(acc[NA - 1][j][2 * i], acc[NA - 1][j][2 * i + 1]), d2);
                                acc[0][j][2 * i] = ga.x;
                                acc[0][j][2 * i + 1] = ga.y;
                                acc[NA - 1][j][2 * i] = gb.x;
                                acc[NA - 1][j][2 * i + 1] = gb.y;
                            } else {
                                av = __fmul2_rn(d2, xh);
                            }
                        } else {
                            ov = __ffma2_rn(x2, nc1, __fmul2_rn(c02, __fmul2_rn(d2, gf[j][i])));
                            if constexpr (ACC_REG) {
                                const float2 ga = __ffma2_rn(__fmul2_rn(d2, x2), c02,
                                                             make_float2(acc[0][j][2 * i], acc[0][j][2 * i + 1]));
                                acc[0][j][2 * i] = ga.x;
                                acc[0][j][2 * i + 1] = ga.y;
                            } else {
                                av = __fmul2_rn(__fmul2_rn(d2, x2), c02);
                            }
                        }
                        o[2 * i] = ov.x;
                        o[2 * i + 1] = ov.y;
                        pa[2 * i] = av.x;
                        pa[2 * i + 1] = av.y;
                        pb[2 * i] = bv.x;
                        pb[2 * i + 1] = bv.y;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float xe = E::get(xv[j], e), de = E::get(dv[j], e), ge = E::get(gv[j], e);
                        if constexpr (LN) {
                            const float xh = (xe - mu) * rs;
                            o[e] = rs * ((de * ge - c0) - xh * c1);
                            if constexpr (ACC_REG) {
                                acc[0][j][e] = fmaf(de, xh, acc[0][j][e]);
                                acc[NA - 1][j][e] += de;
                            } else {
                                pa[e] = de * xh;
                                pb[e] = de;
                            }
                        } else {
                            o[e] = fmaf(-xe, c1, c0 * (de * ge));
                            if constexpr (ACC_REG)
                                acc[0][j][e] = fmaf(de * xe, c0, acc[0][j][e]);
                            else
                                pa[e] = (de * xe) * c0;
                        }
                    }
                }
                O::store(dxr + j * stride, E::pack(o));
#pragma unroll
                for (int k = 0; k < (ACC_REG ? 0 : NA); ++k) {
                    float* d = my_acc + k * slice + j * 32 * VEC;
                    const float* p = k == 0 ? pa : pb;
                    if constexpr (VEC % 4 == 0) {
#pragma unroll
                        for (int e = 0; e < VEC; e += 4) {
                            float4 v = *reinterpret_cast<float4*>(d + e);
                            if constexpr (PAIRS) {
                                const float2 lo = __fadd2_rn(make_float2(v.x, v.y), make_float2(p[e], p[e + 1]));
                                const float2 hi = __fadd2_rn(make_float2(v.z, v.w), make_float2(p[e + 2], p[e + 3]));
                                v = make_float4(lo.x, lo.y, hi.x, hi.y);
                            } else {
                                v.x += p[e];
                                v.y += p[e + 1];
                                v.z += p[e + 2];
                                v.w += p[e + 3];
                            }
                            *reinterpret_cast<float4*>(d + e) = v;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) d[e] += p[e];
                    }
                }
            }
    }

    if constexpr (RING) {
        if (late >= 0 && tid == 0) {
            // Copies still in flight (rows late .. late+stages-1 of this CTA)
            // get one more bounded wait each, so that none lands after this
            // CTA has gone; then tell the host.
            for (int64_t kk = late; kk < late + stages; ++kk)
                if (first_row + kk * row_step < a.M)
                    mbar_wait(&full[kk % stages], static_cast<uint32_t>((kk / stages) & 1));
            atomicAdd(a.wait_timeouts, 1u);
        }
    }

    if constexpr (ACC_REG) {
        // Hand the register accumulators to this thread's shared-memory
        // slots (column positions), where the steps below expect them.
#pragma unroll
        for (int k = 0; k < NA; ++k)
#pragma unroll
            for (int j = 0; j < V; ++j) {
                float* d = my_acc + k * slice + j * 32 * VEC;
                if constexpr (VEC % 4 == 0) {
#pragma unroll
                    for (int e = 0; e < VEC; e += 4)
                        *reinterpret_cast<float4*>(d + e) =
                            make_float4(acc[k][j][e], acc[k][j][e + 1], acc[k][j][e + 2], acc[k][j][e + 3]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) d[e] = acc[k][j][e];
                }
            }
    }

    // Partial rows of the column gradients: one per cluster.
    float* wsp = a.ws + static_cast<int64_t>(blockIdx.x / Q) * NA * N;
    if (C > 1 || Q == 1) {
        // The CTAs of a row's cluster own distinct columns: write them.
#pragma unroll
        for (int k = 0; k < NA; ++k)
#pragma unroll
            for (int j = 0; j < V; ++j)
                if (j < nv) {
                    const float* src = my_acc + k * slice + j * 32 * VEC;
                    float* dst = wsp + k * N + (f0 + j * 32) * VEC;
                    if constexpr (VEC % 4 == 0) {
#pragma unroll
                        for (int e = 0; e < VEC; e += 4)
                            *reinterpret_cast<float4*>(dst + e) = *reinterpret_cast<const float4*>(src + e);
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) dst[e] = src[e];
                    }
                }
        if (C > 1) cluster_barrier();  // no CTA exits while a peer may read its shared memory
    } else {
        // The Q CTAs of this cluster own the same columns (each had its own
        // rows), held at position = column in every CTA's accumulators: CTA
        // q of the cluster adds the Q copies of its share of the columns, in
        // rank order, and writes them.
        cluster_barrier();
        uint32_t peer[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            peer[q] = q < static_cast<int>(Q) ? peer_smem_addr(acc_s, static_cast<uint32_t>(q)) : 0u;
        const int span = (N + static_cast<int>(Q) - 1) / static_cast<int>(Q);
        const int c_lo = static_cast<int>(crank) * span;
        const int c_hi = min(N, c_lo + span);
#pragma unroll
        for (int k = 0; k < NA; ++k)
            for (int c = c_lo + tid; c < c_hi; c += T_) {
                const uint32_t off = static_cast<uint32_t>(k * slice + c) * 4u;
                float s = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < static_cast<int>(Q)) s += ld_peer_f32(peer[q] + off);
                wsp[k * N + c] = s;
            }
        cluster_barrier();  // every peer has read this CTA's accumulators before it exits
    }
}

// Column sums of the partial rows: out_k[c] = sum over p, in order, of
// ws[p][k][c]. With no partial rows (M == 0) the gradients are zero.
template <int NA>
__global__ void __launch_bounds__(256) norm_bwd_colsum(const float* ws, int64_t partials, int32_t N, float* out0,
                                                       float* out1) {
    grid_release();
    grid_wait();
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= N) return;
#pragma unroll
    for (int k = 0; k < NA; ++k) {
        const float* p = ws + k * static_cast<int64_t>(N) + c;
        const int64_t step = static_cast<int64_t>(NA) * N;
        float s = 0.f;
#pragma unroll 8
        for (int64_t i = 0; i < partials; ++i) s += p[i * step];
        (k == 0 ? out0 : out1)[c] = s;
    }
}

// ------------------------------------------------------------ launch
using BwdKernel = void (*)(const BwdArgs);

// Largest accesses per thread a backward variant is built for (registers:
// x, dy and gamma accesses plus the fp32 column accumulators).
constexpr int bwd_vmax(bool ln, int elem_size, int vec) {
    return vec == 1 ? 8 : (ln && elem_size == 2) ? 2 : 4;
}

template <class T, bool LN, int VEC, bool RING>
BwdKernel pick_bwd_r(int V) {
    constexpr int vmax = bwd_vmax(LN, sizeof(T), VEC);
    switch (V) {
        case 1: return norm_bwd_cta<T, VEC, 1, LN, RING>;
        case 2: return vmax >= 2 ? norm_bwd_cta<T, VEC, 2, LN, RING> : nullptr;
        case 4: if constexpr (vmax >= 4) return norm_bwd_cta<T, VEC, 4, LN, RING>; else return nullptr;
        case 8: if constexpr (vmax >= 8) return norm_bwd_cta<T, VEC, 8, LN, RING>; else return nullptr;
        default: return nullptr;
    }
}

// The ring variants exist for 16-byte vector rows only.
template <class T, bool LN, int VEC>
BwdKernel pick_bwd(int V, bool ring) {
    if constexpr (VEC > 1) {
        if (ring) return pick_bwd_r<T, LN, VEC, true>(V);
    }
    return ring ? nullptr : pick_bwd_r<T, LN, VEC, false>(V);
}

inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, unsigned cluster,
                              cudaStream_t stream, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// CTAs of `k` (with `threads` threads, `smem` bytes of dynamic shared memory,
// launched in clusters of `q`) that can be resident on device `dev` at
// once, a multiple of q; queried once per configuration and device. Also
// opts the kernel in to the device's largest dynamic shared memory when it
// needs more than 48 KB.
inline cudaError_t bwd_resident_ctas(BwdKernel k, int threads, size_t smem, int q, int dev, int num_sms,
                                     int64_t* out) {
    struct Key {
        const void* fn;
        int threads, q, dev;
        size_t smem;
        bool operator<(const Key& o) const {
            return std::tie(fn, threads, q, dev, smem) < std::tie(o.fn, o.threads, o.q, o.dev, o.smem);
        }
    };
    static std::mutex mu;
    static std::map<Key, int64_t> cache;
    const Key key{reinterpret_cast<const void*>(k), threads, q, dev, smem};
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    if (smem > 48 * 1024) {
        // Opt in to the device's largest dynamic shared memory per block (not
        // just this configuration's: another configuration of the same
        // kernel must never lower the limit below what a cached one needs).
        int optin = 0;
        cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(k));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(k), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
    }
    int64_t ctas = 0;
    if (q > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(q));
        cfg.blockDim = dim3(static_cast<unsigned>(threads));
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(q);
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(k), &cfg);
        if (e != cudaSuccess) return e;
        ctas = static_cast<int64_t>(n) * q;
    } else {
        int n = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reinterpret_cast<const void*>(k),
                                                                            threads, smem);
        if (e != cudaSuccess) return e;
        ctas = static_cast<int64_t>(n) * num_sms;
    }
    cache[key] = ctas;
    *out = ctas;
    return cudaSuccess;
}

// The plan has been validated on the host (one round covers the row; grid a
// multiple of the cluster; `group` = launched cluster size). `grid` is an
// upper bound: the launch takes no more CTAs than can be resident at once
// (the grid-stride loop covers the rows either way), and the column sums
// read only the partial rows that were written.
template <class T, bool LN>
cudaError_t launch_norm_bwd(const norm_plan& p, const BwdArgs& a, cudaStream_t stream, int dev, int num_sms) {
    int64_t grid = 0;
    if (a.M > 0 && p.grid > 0) {
        const bool ring = p.stages > 0;
        const BwdKernel k = p.vec_elems == 1 ? pick_bwd<T, LN, 1>(p.per_thread, ring)
                                             : pick_bwd<T, LN, ElemVec<T>::value>(p.per_thread, ring);
        if (k == nullptr) return cudaErrorInvalidValue;
        const size_t smem = static_cast<size_t>(bwd_smem_bytes(LN, p.threads, p.per_thread, p.vec_elems, p.stages));
        int64_t resident = 0;
        const cudaError_t e0 = bwd_resident_ctas(k, p.threads, smem, p.group, dev, num_sms, &resident);
        if (e0 != cudaSuccess) return e0;
        if (resident < p.group) return cudaErrorInvalidConfiguration;  // not even one cluster fits
        grid = std::min<int64_t>(p.grid, resident);
        BwdArgs args = a;
        args.stages = p.stages;
        if (ring) {
            args.wait_timeouts = wait_counter(dev);
            if (args.wait_timeouts == nullptr) return cudaErrorInvalidSymbol;
        }
        void* kargs[] = {&args};
        const cudaError_t e = launch_pdl(reinterpret_cast<const void*>(k), dim3(static_cast<unsigned>(grid)),
                                         dim3(static_cast<unsigned>(p.threads)), smem,
                                         static_cast<unsigned>(p.group), stream, kargs);
        if (e != cudaSuccess) return e;
    }
    const float* ws = a.ws;
    int64_t parts = grid / p.group;
    int32_t N = a.N;
    float* o0 = a.dgamma;
    float* o1 = LN ? a.dbeta : a.dgamma;
    void* cargs[] = {&ws, &parts, &N, &o0, &o1};
    return launch_pdl(reinterpret_cast<const void*>(norm_bwd_colsum<LN ? 2 : 1>),
                      dim3(static_cast<unsigned>((N + 255) / 256)), dim3(256), 0, 1, stream, cargs);
}

}  // namespace libnorm
