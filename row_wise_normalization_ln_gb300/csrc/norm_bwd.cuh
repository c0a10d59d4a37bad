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

// ------------------------------------------------------------ row arithmetic
// The per-row work of a thread, shared by the backward kernels: its gamma
// (w) slice, its column accumulators and the two passes over one row's
// accesses (the pair of row sums; then dx and the column terms).
//
// The column accumulators live in registers (in this thread's shared-memory
// slots for the 16-bit variants of 4 accesses per thread); at the end they
// go to dynamic shared memory, [NA][T*V*VEC] floats, each thread at the
// positions of its own columns.
template <class T, int VEC, int V, bool LN>
struct BwdRow {
    using O = OpsFor<T, VEC>;
    using E = BwdElem<T, VEC>;
    using Raw = typename O::Raw;
    using P = typename PairOf<T>::type;
    static constexpr int NA = LN ? 2 : 1;
    // 16-bit rows work on fp32 pairs with the packed instructions and keep
    // gamma widened (gf); other rows work on scalars.
    static constexpr bool PAIRS = VEC == 8;
    static constexpr bool ACC_REG = !(VEC == 8 && V >= 4);

    Raw gv[V];
    float2 gf[PAIRS ? V : 1][4];
    float acc[ACC_REG ? NA : 1][ACC_REG ? V : 1][ACC_REG ? VEC : 1];
    float* my_acc;  // this thread's first accumulator slot in shared memory
    int slice;      // floats per shared-memory accumulator array

    __device__ __forceinline__ void init(const T* gp, int stride, int nv, float* acc_slot, int slice_floats) {
        my_acc = acc_slot;
        slice = slice_floats;
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

    // This thread's share of the row's pair of sums: LayerNorm (sum g,
    // sum g * xhat) with g = dy * gamma, xhat = (x - mean) * rstd; RMSNorm
    // (sum x^2, sum dy * w * x).
    __device__ __forceinline__ float2 partials(const Raw (&xv)[V], const Raw (&dv)[V], int nv, float mu,
                                               float rs) const {
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
        return make_float2(s0, s1);
    }

    // dx of the row from its pair of sums S, stored at dxr (this thread's
    // first access), and the row's terms added to the column accumulators.
    __device__ __forceinline__ void output(const Raw (&xv)[V], const Raw (&dv)[V], int nv, float mu, float rs,
                                           float2 S, float invN, float eps, T* dxr, int stride) {
        float c0, c1;  // LayerNorm: mean(g), mean(g xhat); RMSNorm: rstd, rstd^3 mean(dy w x)
        if constexpr (LN) {
            c0 = S.x * invN;
            c1 = S.y * invN;
        } else {
            c0 = rsqrtf(S.x * invN + eps);
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
                                const float2 ga =
                                    __ffma2_rn(d2, xh, make_float2(acc[0][j][2 * i], acc[0][j][2 * i + 1]));
                                const float2 gb =
                                    __fadd2_rn(make_float2(acc[NA - 1][j][2 * i], acc[NA - 1][j][2 * i + 1]), d2);
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
                                const float2 hi =
                                    __fadd2_rn(make_float2(v.z, v.w), make_float2(p[e + 2], p[e + 3]));
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

    // Hand the register accumulators to this thread's shared-memory slots
    // (column positions), where the column-sum steps expect them.
    __device__ __forceinline__ void acc_to_smem() const {
        if constexpr (ACC_REG) {
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
    }
};

// The end of every backward kernel: the CTA's column accumulators (in shared
// memory at acc_s, [NA][slice] floats) become partial rows of the
// workspace, one per launched cluster of Q CTAs. The CTAs of a row's cluster
// (C > 1) own distinct columns and write them; the Q CTAs of a reduction
// cluster (C == 1) own the same columns, and CTA q adds the Q copies of its
// share of them in rank order. Ends with the cluster's last barrier.
template <int VEC, int V, int NA>
__device__ __forceinline__ void write_partials(const BwdArgs& a, const float* acc_s, int slice, int C, int f0, int nv) {
    const int N = a.N;
    const int T_ = blockDim.x;
    const int tid = threadIdx.x;
    const int local = (tid >> 5) * V * 32 + (tid & 31);
    const float* my_acc = acc_s + local * VEC;
    const uint32_t Q = cluster_size();
    const uint32_t crank = cluster_rank();
    float* wsp = a.ws + static_cast<int64_t>(blockIdx.x / Q) * NA * N;
    if (C > 1 || Q == 1) {
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

// Rows over a cluster (C > 1): the row's pair of sums meets without a
// cluster barrier (whose release waited for every earlier store of the CTA,
// the row's dx included, to reach L2). Each CTA reduces its pair in shared
// memory; thread 0 then sends it to every CTA of the cluster with an
// asynchronous store counted on that CTA's mbarrier (slot [rank]), and
// announces the C pairs it expects on its own. Every thread waits for the
// phase and adds the C pairs in rank order. Slots and barriers alternate by
// row parity: a CTA sends a row's pair only after its wait on the previous
// row, which needs every peer's pair of that row, which each peer sends
// only after reading the pairs of the row before.
struct ClusterPairSmem {
    float2 part[2][8];
    uint64_t bar[2];
};

__device__ __forceinline__ float2 cluster_row_sum2(PairReduceSmem& red, ClusterPairSmem& cred, int it, float2 v,
                                                   int C, int rank, int nwarps, int wwidth, uint64_t limit,
                                                   bool& late) {
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int s = it & 1;
    v.x = group_sum(v.x, 32);
    v.y = group_sum(v.y, 32);
    if (lane == 0) red.warp_part[s][tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
        float2 w = lane < nwarps ? red.warp_part[s][lane] : make_float2(0.f, 0.f);
        w.x = sum_first_lanes(w.x, wwidth);
        w.y = sum_first_lanes(w.y, wwidth);
        if (tid == 0) {
            mbar_arrive_expect(&cred.bar[s], static_cast<uint32_t>(C) * 8u);
            for (int q = 0; q < C; ++q)
                st_async_peer_f32x2(peer_smem_addr(&cred.part[s][rank], static_cast<uint32_t>(q)), w,
                                    peer_smem_addr(&cred.bar[s], static_cast<uint32_t>(q)));
        }
    }
    if (!mbar_wait(&cred.bar[s], static_cast<uint32_t>((it >> 1) & 1), limit)) late = true;
    const float2 p = lane < C ? cred.part[s][lane] : make_float2(0.f, 0.f);
    return make_float2(sum_first_lanes(p.x, C), sum_first_lanes(p.y, C));
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
// it.
// CL: launched for rows over a cluster (row_cluster > 1); the kernels for
// one CTA per row carry none of the cluster code.
template <class T, int VEC, int V, bool LN, bool RING, bool CL>
__global__ void __launch_bounds__(kBwdMaxThreads) norm_bwd_cta(const BwdArgs a) {
    static_assert(!RING || VEC > 1, "the ring moves 16-byte vectors");
    using R = BwdRow<T, VEC, V, LN>;
    using O = typename R::O;
    using Raw = typename R::Raw;
    constexpr int NA = R::NA;
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
    const int C = CL ? a.row_cluster : 1;
    const int rank = C > 1 ? static_cast<int>(cluster_rank()) : 0;
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
    // RING: `stages` stages of this CTA's slices of an upcoming row, x then
    // dy (V*T 16-byte slots each), then one mbarrier per stage; after the
    // shared-memory accumulators, or over them when the accumulators are in
    // registers until the end (they reach their slots after the last row).
    const int stages = RING ? a.stages : 0;
    uint4* ring = reinterpret_cast<uint4*>(acc_s + (R::ACC_REG ? 0 : NA * slice));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + 2 * stages * V * T_);

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
    // RING: set by any thread whose wait for a stage ran out; read by every
    // thread before its next wait and by thread 0 before its next copy, each
    // after the barrier of the row's pair reduction, so that from the row
    // after a timeout on the whole CTA neither waits nor copies.
    __shared__ int s_late;
    __shared__ std::conditional_t<CL, ClusterPairSmem, char> cred;  // rows over a cluster
    if (RING || CL) {
        if (tid == 0) {
            if (RING) {
                for (int k = 0; k < stages; ++k) mbar_init(&full[k], 1);
                s_late = 0;
            }
            if constexpr (CL) {
                mbar_init(&cred.bar[0], 1);
                mbar_init(&cred.bar[1], 1);
            }
            mbar_init_fence();
        }
        // Every barrier is initialised before any CTA of the cluster
        // addresses it.
        if constexpr (CL)
            cluster_barrier();
        else
            __syncthreads();
    }

    grid_release();
    grid_wait();
    const uint64_t limit = (RING || CL) ? a.wait->limit_ns : 0;
    bool rlate = false;  // CL: a wait for the row's pairs ran out (the outputs are then void)

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
    int64_t issued = 0;  // RING, thread 0: rows of this CTA whose copies it issued
    if constexpr (RING) {
        if (tid == 0)
            for (int k = 0; k < stages; ++k)
                if (first_row + k * row_step < a.M) {
                    issue(first_row + k * row_step, k);
                    ++issued;
                }
    }

    R rw;
    rw.init(static_cast<const T*>(a.gamma) + f0 * VEC, stride, nv, acc_s + local * VEC, slice);
    const T* xbase = static_cast<const T*>(a.x) + f0 * VEC;
    const T* dybase = static_cast<const T*>(a.dy) + f0 * VEC;

    // LayerNorm: the row's mean and rstd. Without a ring they are loaded a
    // row ahead (a load at the row's start would stall all of its
    // arithmetic on an L2 round trip); with one, at the row's start, before
    // the wait for its stage.
    float2 ms = make_float2(0.f, 0.f);
    if constexpr (LN && !RING) {
        if (first_row < a.M) ms = make_float2(a.mean[first_row], a.rstd[first_row]);
    }
    int it = 0;
    int st = 0;            // RING: this row's stage
    uint32_t parity = 0;   // ... and the phase parity to wait for
    volatile int& late = s_late;
    int64_t seen = 0;      // RING, thread 0: leading rows whose copies it saw complete
    bool waiting = true;   // RING: this thread still waits for its stages
    for (int64_t row = first_row; row < a.M; row += row_step, ++it) {
        if (tid == 0) prefetch_row(row + ahead * row_step);
        Raw xv[V], dv[V];
        if constexpr (RING) {
            // The row's statistics: loaded here, their latency hidden behind
            // the wait for the row's stage.
            if constexpr (LN) ms = make_float2(a.mean[row], a.rstd[row]);
            // After a wait has run out the CTA neither waits nor copies any
            // more (its outputs are void by then); the kernel still ends.
            if (waiting) {
                if (late)
                    waiting = false;
                else if (!mbar_wait(&full[st], parity, limit))
                    late = 1, waiting = false;
                else
                    seen = it + 1;
            }
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
        const float mu = ms.x, rs = ms.y;
        const float2 pr = rw.partials(xv, dv, nv, mu, rs);
        float2 S;
        if constexpr (CL)
            S = cluster_row_sum2(red, cred, it, pr, C, rank, nwarps, wwidth, limit, rlate);
        else
            S = row_sum2(red, it & 1, pr, 1, nwarps, wwidth);
        // Without a ring: the next row's statistics, issued after the row's
        // block barrier (a barrier would wait for a load issued before it)
        // and needed only after this row's output pass.
        if constexpr (LN && !RING) {
            if (row + row_step < a.M) ms = make_float2(a.mean[row + row_step], a.rstd[row + row_step]);
        }
        if constexpr (RING) {
            // Every thread has read this stage before the barrier above:
            // refill it with the row `stages` turns ahead.
            if (tid == 0 && !late && row + stages * row_step < a.M) {
                fence_proxy_async();
                issue(row + stages * row_step, st);
                ++issued;
            }
            if (++st == stages) st = 0, parity ^= 1u;
        }
        rw.output(xv, dv, nv, mu, rs, S, invN, a.eps, static_cast<T*>(a.dx) + row * N + f0 * VEC, stride);
    }

    if constexpr (RING) {
        if (tid == 0 && late) {
            // Copies that may still be in flight (the rows issued after the
            // last one thread 0 saw complete; a stage is refilled only after
            // its previous row completed) get one more wait each, with the
            // full limit, so that none lands after this CTA has gone; then
            // tell the host.
            for (int64_t kk = seen; kk < issued; ++kk)
                mbar_wait(&full[kk % stages], static_cast<uint32_t>((kk / stages) & 1), kDefaultWaitLimitNs);
            atomicAdd(&a.wait->timeouts, 1u);
        }
    }
    // With register accumulators the ring overlaps their shared-memory
    // slots: every thread is past its last read of the ring (and thread 0
    // past its drain) before any slot is written.
    if constexpr (CL) {
        if (__syncthreads_or(rlate) && tid == 0) atomicAdd(&a.wait->timeouts, 1u);
    } else {
        __syncthreads();
    }
    rw.acc_to_smem();
    write_partials<VEC, V, NA>(a, acc_s, slice, C, f0, nv);
}

// ------------------------------------------------------------ register pipeline
// The backward for rows that one CTA covers (row_cluster == 1), with the
// next row's loads in flight while the current row is reduced and written.
// Each thread holds two register sets of its x and dy slices (and the row's
// mean and rstd) and alternates between them (the loop body is unrolled
// twice, so no register is copied): it loads row r + step into one set right
// after it has handed in its share of row r's sums, while the other set
// still holds row r for the output pass. Lane 0 of each warp stores the
// warp's pair; then every thread issues its next loads and meets the others,
// at a block barrier (CTAs of 8 or more warps) or on an mbarrier (lane 0
// arrives with release before the loads, every thread waits with acquire
// after them), and reads the pairs. Rows three steps ahead are still
// bulk-prefetched into L2, so the register loads are L2 hits.
//
// Slots and barriers alternate by row parity. A warp writes a row's pair
// only after it has passed the previous row's meeting, which every warp
// reaches only after reading the pairs of the row before; so a slot is
// rewritten only after all its readers are done, and an mbarrier phase
// never completes twice ahead of a waiter.
struct PipeReduceSmem {
    float2 warp_part[2][32];
    uint64_t bar[2];
};

// BAR: the warps meet at a block barrier and x and dy are loaded without
// allocating in L1 (launched for CTAs of 8 or more warps); otherwise the
// warps meet on the mbarrier and the loads are plain.
template <class T, int VEC, int V, bool LN, bool BAR>
__global__ void __launch_bounds__(kBwdMaxThreads) norm_bwd_pipe(const BwdArgs a) {
    using R = BwdRow<T, VEC, V, LN>;
    using O = typename R::O;
    using Raw = typename R::Raw;
    constexpr int NA = R::NA;
    __shared__ PipeReduceSmem red;
    extern __shared__ float4 acc_v[];
    float* acc_s = reinterpret_cast<float*>(acc_v);

    const int T_ = blockDim.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T_ >> 5;
    int wwidth = 1;
    while (wwidth < nwarps) wwidth <<= 1;
    const int64_t first_row = blockIdx.x;
    const int64_t row_step = gridDim.x;
    const int N = a.N;
    const int nacc = (N + VEC - 1) / VEC;
    const int stride = 32 * VEC;
    const int local = warp * V * 32 + lane;  // first access within the row
    const int nv = valid_runs(nacc, local, 32, V);
    const float invN = 1.f / static_cast<float>(N);
    const int slice = T_ * V * VEC;

    const uint32_t row_bytes = static_cast<uint32_t>(N * sizeof(T));
    auto prefetch_row = [&](int64_t r) {
        if (r >= a.M) return;
        if constexpr (VEC > 1) {
            prefetch_l2_bulk(static_cast<const T*>(a.x) + r * N, row_bytes);
            prefetch_l2_bulk(static_cast<const T*>(a.dy) + r * N, row_bytes);
        }
        if constexpr (LN) {
            prefetch_l2_line(a.mean + r);
            prefetch_l2_line(a.rstd + r);
        }
    };
    if (tid == 0) {
        for (int k = 0; k < 3; ++k) prefetch_row(first_row + k * row_step);
        mbar_init(&red.bar[0], nwarps);
        mbar_init(&red.bar[1], nwarps);
    }
    __syncthreads();
    grid_release();
    grid_wait();
    const uint64_t limit = a.wait->limit_ns;
    bool late = false;  // a wait for the row's sums ran out (the outputs are then void)

    R rw;
    rw.init(static_cast<const T*>(a.gamma) + local * VEC, stride, nv, acc_s + local * VEC, slice);
    const T* xbase = static_cast<const T*>(a.x) + local * VEC;
    const T* dybase = static_cast<const T*>(a.dy) + local * VEC;

    // A row's slices of x and dy and (LayerNorm) its mean and rstd. CTAs of
    // 8 or more warps (BAR) load them without allocating in L1 (A/B on
    // GB300: LayerNorm bf16 4096x8192 38.2 -> 37.3 us, 4096x4096 23.0 ->
    // 22.6 us; the 4-warp CTAs of 2048-wide rows lose 1 to 5 % with it).
    auto load = [&](Raw (&xv)[V], Raw (&dv)[V], float2& ms, int64_t row) {
        if (row >= a.M) return;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nv) {
                xv[j] = BAR ? O::load_stream(xbase + row * N + j * stride) : O::load(xbase + row * N + j * stride);
                dv[j] = BAR ? O::load_stream(dybase + row * N + j * stride) : O::load(dybase + row * N + j * stride);
            }
        if constexpr (LN) ms = make_float2(a.mean[row], a.rstd[row]);
    };
    // One row: its sums handed in, the next row's loads issued into the
    // other set, the sums collected, dx written.
    auto step = [&](Raw (&xc)[V], Raw (&dc)[V], float2& mc, Raw (&xn)[V], Raw (&dn)[V], float2& mn, int64_t row,
                    int it) {
        if (tid == 0) prefetch_row(row + 3 * row_step);
        const float mu = mc.x, rs = mc.y;
        float2 p = rw.partials(xc, dc, nv, mu, rs);
        p.x = group_sum(p.x, 32);
        p.y = group_sum(p.y, 32);
        const int s = it & 1;
        if (lane == 0) {
            red.warp_part[s][warp] = p;
            if constexpr (!BAR) mbar_arrive(&red.bar[s]);
        }
        load(xn, dn, mn, row + row_step);
        if constexpr (BAR) {
            __syncthreads();
        } else {
            // Every warp of the CTA arrives once per row, so the phase
            // completes; the wait is bounded all the same (the device's
            // wait limit).
            if (!mbar_wait(&red.bar[s], static_cast<uint32_t>((it >> 1) & 1), limit)) late = true;
        }
        float2 w = lane < nwarps ? red.warp_part[s][lane] : make_float2(0.f, 0.f);
        w.x = sum_first_lanes(w.x, wwidth);
        w.y = sum_first_lanes(w.y, wwidth);
        rw.output(xc, dc, nv, mu, rs, w, invN, a.eps, static_cast<T*>(a.dx) + row * N + local * VEC, stride);
    };

    Raw xa[V], da[V], xb[V], db[V];
    float2 ma = make_float2(0.f, 0.f), mb = ma;  // (mean, rstd) of the rows in xa/da and xb/db
    load(xa, da, ma, first_row);
    int it = 0;
    for (int64_t row = first_row; row < a.M; row += 2 * row_step, it += 2) {
        step(xa, da, ma, xb, db, mb, row, it);
        if (row + row_step >= a.M) break;
        step(xb, db, mb, xa, da, ma, row + row_step, it + 1);
    }
    if (__syncthreads_or(late) && tid == 0) atomicAdd(&a.wait->timeouts, 1u);
    rw.acc_to_smem();
    write_partials<VEC, V, NA>(a, acc_s, slice, 1, local, nv);
}

// Column sums of the partial rows: out_k[c] = sum over p of ws[p][k][c]. A
// CTA of kWarps warps (8, or 32 for more than 64 partial rows) covers 32*W
// columns (W consecutive columns per lane, one W-wide load per partial
// row): warp w adds partial rows w, w+kWarps, w+2*kWarps, ... in that order,
// then the warp sums of each column are added in warp order. The order
// depends only on the number of partial rows, so the result is
// deterministic for a plan; the partial rows are read by many warps at once,
// each with several loads in flight and few rows in its chain. With no
// partial rows (M == 0) the gradients are zero. W = 4 needs N % 4 == 0
// (16-byte aligned partial rows).
template <int NA, int W, int kWarps>
__global__ void __launch_bounds__(kWarps * 32) norm_bwd_colsum(const float* ws, int64_t partials, int32_t N,
                                                               float* out0, float* out1) {
    constexpr int kCols = 32 * W;
    __shared__ float part[NA][kWarps][kCols];
    grid_release();
    grid_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t cbase = static_cast<int64_t>(blockIdx.x) * kCols;
    const int64_t c0 = cbase + lane * W;  // this lane's first column
    const int64_t step = static_cast<int64_t>(NA) * N;
    float s[NA][W];
#pragma unroll
    for (int k = 0; k < NA; ++k)
#pragma unroll
        for (int e = 0; e < W; ++e) s[k][e] = 0.f;
    if (c0 < N) {
#pragma unroll 4
        for (int64_t p = warp; p < partials; p += kWarps) {
#pragma unroll
            for (int k = 0; k < NA; ++k) {
                const float* src = ws + p * step + k * static_cast<int64_t>(N) + c0;
                if constexpr (W == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(src);
                    s[k][0] += v.x;
                    s[k][1] += v.y;
                    s[k][2] += v.z;
                    s[k][3] += v.w;
                } else {
                    s[k][0] += *src;
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < NA; ++k)
#pragma unroll
        for (int e = 0; e < W; ++e) part[k][warp][lane * W + e] = s[k][e];
    __syncthreads();
    for (int i = threadIdx.x; i < NA * kCols; i += blockDim.x) {
        const int k = i / kCols;
        const int cc = i - k * kCols;
        const int64_t c = cbase + cc;
        if (c < N) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) t += part[k][w][cc];
            (k == 0 ? out0 : out1)[c] = t;
        }
    }
}

// ------------------------------------------------------------ launch
using BwdKernel = void (*)(const BwdArgs);

// Largest accesses per thread a backward variant is built for (registers:
// x, dy and gamma accesses plus the fp32 column accumulators).
constexpr int bwd_vmax(bool ln, int elem_size, int vec) {
    return vec == 1 ? 8 : (ln && elem_size == 2) ? 2 : 4;
}

template <class T, bool LN, int VEC, bool RING, bool CL>
BwdKernel pick_bwd_c(int V) {
    constexpr int vmax = bwd_vmax(LN, sizeof(T), VEC);
    switch (V) {
        case 1: return norm_bwd_cta<T, VEC, 1, LN, RING, CL>;
        case 2: return vmax >= 2 ? norm_bwd_cta<T, VEC, 2, LN, RING, CL> : nullptr;
        case 4: if constexpr (vmax >= 4) return norm_bwd_cta<T, VEC, 4, LN, RING, CL>; else return nullptr;
        case 8: if constexpr (vmax >= 8) return norm_bwd_cta<T, VEC, 8, LN, RING, CL>; else return nullptr;
        default: return nullptr;
    }
}

template <class T, bool LN, int VEC, bool RING>
BwdKernel pick_bwd_r(int V, bool cl) {
    return cl ? pick_bwd_c<T, LN, VEC, RING, true>(V) : pick_bwd_c<T, LN, VEC, RING, false>(V);
}

template <class T, bool LN, int VEC, bool BAR>
BwdKernel pick_bwd_pipe_b(int V) {
    constexpr int vmax = bwd_vmax(LN, sizeof(T), VEC);
    switch (V) {
        case 1: return norm_bwd_pipe<T, VEC, 1, LN, BAR>;
        case 2: return vmax >= 2 ? norm_bwd_pipe<T, VEC, 2, LN, BAR> : nullptr;
        case 4: if constexpr (vmax >= 4) return norm_bwd_pipe<T, VEC, 4, LN, BAR>; else return nullptr;
        case 8: if constexpr (vmax >= 8) return norm_bwd_pipe<T, VEC, 8, LN, BAR>; else return nullptr;
        default: return nullptr;
    }
}

// CTAs of 8 or more warps meet at a block barrier, smaller ones on the
// mbarrier (measured on GB300: LayerNorm bf16 4096x8192, 512 threads, 42.3 us
// with the mbarrier and 40.7 with the block barrier; RMSNorm bf16 65536x2048,
// 128 threads, 126.5 and 135.2 us).
template <class T, bool LN, int VEC>
BwdKernel pick_bwd_pipe(int V, int threads) {
    return threads >= 256 ? pick_bwd_pipe_b<T, LN, VEC, true>(V) : pick_bwd_pipe_b<T, LN, VEC, false>(V);
}

// stages 0: rows from L2 after a bulk prefetch; 1: the register pipeline;
// 2..4: the shared-memory ring (16-byte vector rows only). `cl`: rows over
// a cluster of CTAs.
template <class T, bool LN, int VEC>
BwdKernel pick_bwd(int V, int stages, bool cl, int threads) {
    if (stages == 1) return cl ? nullptr : pick_bwd_pipe<T, LN, VEC>(V, threads);
    if constexpr (VEC > 1) {
        if (stages >= 2) return pick_bwd_r<T, LN, VEC, true>(V, cl);
    }
    return stages >= 2 ? nullptr : pick_bwd_r<T, LN, VEC, false>(V, cl);
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
        const bool cl = p.cluster > 1;
        const BwdKernel k = p.vec_elems == 1
                                ? pick_bwd<T, LN, 1>(p.per_thread, p.stages, cl, p.threads)
                                : pick_bwd<T, LN, ElemVec<T>::value>(p.per_thread, p.stages, cl, p.threads);
        if (k == nullptr) return cudaErrorInvalidValue;
        const size_t smem = static_cast<size_t>(bwd_smem_bytes(LN, p.threads, p.per_thread, p.vec_elems, p.stages));
        int64_t resident = 0;
        const cudaError_t e0 = bwd_resident_ctas(k, p.threads, smem, p.group, dev, num_sms, &resident);
        if (e0 != cudaSuccess) return e0;
        if (resident < p.group) return cudaErrorInvalidConfiguration;  // not even one cluster fits
        grid = std::min<int64_t>(p.grid, resident);
        BwdArgs args = a;
        args.stages = p.stages;
        args.wait = wait_state(dev);
        if (args.wait == nullptr) return cudaErrorInvalidSymbol;
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
    constexpr int NA = LN ? 2 : 1;
    const bool wide = N % 4 == 0 && (reinterpret_cast<uintptr_t>(ws) & 15u) == 0;
    const int cols = wide ? 128 : 32;
    // Many partial rows (every CTA of a persistent grid writes its own):
    // 32 warps per CTA, so that no warp walks more than a few of them
    // (LayerNorm bf16 4096x8192 backward with 152 partial rows: 42.8 -> 38.0
    // us).
    const bool many = parts > 64;
    const void* fn = wide ? (many ? reinterpret_cast<const void*>(norm_bwd_colsum<NA, 4, 32>)
                                  : reinterpret_cast<const void*>(norm_bwd_colsum<NA, 4, 8>))
                          : (many ? reinterpret_cast<const void*>(norm_bwd_colsum<NA, 1, 32>)
                                  : reinterpret_cast<const void*>(norm_bwd_colsum<NA, 1, 8>));
    return launch_pdl(fn, dim3(static_cast<unsigned>((N + cols - 1) / cols)), dim3(many ? 1024 : 256), 0, 1, stream,
                      cargs);
}

}  // namespace libnorm
