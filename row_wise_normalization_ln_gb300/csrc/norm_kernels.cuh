// Row-wise LayerNorm / RMSNorm forward kernels for sm_103a.
//
// Both kernels read x from HBM once, keep the row in registers, reduce the
// statistics in fp32 and write y in the same pass (fused affine and cast):
//
//   norm_fwd_group  `group` lanes of a warp own a row (short rows). The
//                   statistics meet in a xor-shuffle butterfly.
//   norm_fwd_cta    a CTA, or a cluster of CTAs, owns a row (long rows).
//                   Warp butterflies, then shared memory across warps, then
//                   distributed shared memory across the cluster.
//
// LayerNorm statistics are Welford states ([Ch7] §7.4): each thread forms
// (n, mean, M2) of its own register-resident elements, shifted by the row's
// first element, by a two-pass over its registers ([T3] §② trap 2: the row
// is in registers, so "two passes" cost no extra memory traffic), and the
// states are merged with the parallel rule of [Ch7] §7.4.1. The variance is never formed as E[x^2] - E[x]^2. Elements
// beyond N are never loaded and never counted ([T3] §② trap 1).
//
// Sources (page title, section):
//   [Ch7] "第 7 章 LayerNorm 与 RMSNorm": §7.1, §7.4-7.6.
//   [T3]  "T3 讲解：LayerNorm / RMSNorm 的 forward": §②, §③.
#pragma once

#include "norm_args.h"
#include "norm_device.cuh"

namespace libnorm {

template <class T>
struct ElemVec {
    static constexpr int value = 16 / sizeof(T);
};

// (n, mean, M2) of this thread's valid elements, two-pass over registers,
// on the row shifted by K (the row's first element, the same for every
// thread of the row): the variance does not change under a shift, the
// differences x - K of nearby fp32 values are exact, and the merged means
// stay small, so a row whose mean dwarfs its spread ([Ch7] §7.3) keeps its
// digits through every merge. The returned mean is the mean of x - K.
template <class T, int VEC, int V>
__device__ __forceinline__ Welford thread_welford(const Frag<T, VEC> (&f)[V], const bool (&ok)[V], float K) {
    float sum = 0.f;
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < V; ++j)
        if (ok[j]) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) sum += f[j].get(e) - K;
            cnt += VEC;
        }
    if (cnt == 0) return welford_empty();
    const float n = static_cast<float>(cnt);
    const float mu = sum / n;
    float m2 = 0.f;
#pragma unroll
    for (int j = 0; j < V; ++j)
        if (ok[j]) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float d = (f[j].get(e) - K) - mu;
                m2 = fmaf(d, d, m2);
            }
        }
    return {n, mu, m2};
}

// Sum of squares of this thread's valid elements (RMSNorm, [Ch7] §7.5.1).
template <class T, int VEC, int V>
__device__ __forceinline__ float thread_sumsq(const Frag<T, VEC> (&f)[V], const bool (&ok)[V]) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < V; ++j)
        if (ok[j]) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss = fmaf(f[j].get(e), f[j].get(e), ss);
        }
    return ss;
}

// Normalise, apply the affine parameters, round and store one access.
// LayerNorm: y = ((x - K) - mu) * rstd * gamma + beta, where mu is the mean
// of the shifted row (so x - mean is formed without the rounding of the
// fp32 mean); RMSNorm: y = x * rstd * w.
template <class T, int VEC, bool LN>
__device__ __forceinline__ void emit(const Frag<T, VEC>& xf, const T* gamma, const T* beta, T* y,
                                     int elem, float K, float mu, float rs) {
    Frag<T, VEC> g;
    g.load_param(gamma + elem);
    float o[VEC];
    if constexpr (LN) {
        Frag<T, VEC> b;
        b.load_param(beta + elem);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = fmaf(((xf.get(e) - K) - mu) * rs, g.get(e), b.get(e));
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = (xf.get(e) * rs) * g.get(e);
    }
    Frag<T, VEC>::store(y + elem, o);
}

// ------------------------------------------------------------------ GROUP
// Lanes [k*G, (k+1)*G) of the CTA own row blockIdx*rows_per_cta + k. Lane l
// of a group holds accesses l, l+G, l+2G, ... of the row (coalesced: the G
// lanes of a group read G consecutive accesses per instruction).
template <class T, int VEC, int V, bool LN>
__global__ void __launch_bounds__(1024) norm_fwd_group(const NormArgs a) {
    const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
    const T* __restrict__ beta = static_cast<const T*>(a.beta);
    const int G = a.group;
    const int tid = threadIdx.x;
    const int gl = tid & (G - 1);
    const int rows_per_cta = blockDim.x / G;
    const int nacc = (a.N + VEC - 1) / VEC;

    for (int64_t rb = blockIdx.x; rb * rows_per_cta < a.M; rb += gridDim.x) {
        const int64_t row = rb * rows_per_cta + tid / G;
        const bool row_ok = row < a.M;
        const T* xr = static_cast<const T*>(a.x) + row * a.N;
        T* yr = static_cast<T*>(a.y) + row * a.N;

        Frag<T, VEC> f[V];
        bool ok[V];
        float K = 0.f;
        if (LN && row_ok) {
            Frag<T, 1> k0;
            k0.load(xr);
            K = k0.get(0);
        }
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int acc = j * G + gl;
            ok[j] = row_ok && acc < nacc;
            if (ok[j]) f[j].load(xr + acc * VEC);
        }

        float mu = 0.f, rs;
        if constexpr (LN) {
            const Welford s = group_merge(thread_welford<T, VEC, V>(f, ok, K), G);
            mu = s.mean;
            rs = rsqrtf(s.m2 / static_cast<float>(a.N) + a.eps);
            if (gl == 0 && row_ok) {
                if (a.mean) a.mean[row] = K + mu;
                if (a.rstd) a.rstd[row] = rs;
            }
        } else {
            const float ss = group_sum(thread_sumsq<T, VEC, V>(f, ok), G);
            rs = rsqrtf(ss / static_cast<float>(a.N) + a.eps);
        }
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (ok[j]) emit<T, VEC, LN>(f[j], gamma, beta, yr, (j * G + gl) * VEC, K, mu, rs);
    }
}

// -------------------------------------------------------------------- CTA
// A cluster of C CTAs (C = 1 without a cluster launch) owns one row per
// iteration. In round r, thread t of CTA rank k holds accesses
// ((r*C + k)*V + j)*T + t for j < V. With one round the row stays in
// registers from load to store. With several rounds every round is read for
// the statistics; the output pass then walks the rounds backwards, reusing
// the registers of the last round and re-reading the others.
template <class T, int VEC, int V, bool LN>
__global__ void __launch_bounds__(1024) norm_fwd_cta(const NormArgs a) {
    __shared__ float warp_part[2][3][32];  // per-warp states, double-buffered by row parity
    __shared__ float cta_part[2][3];       // this CTA's state, read by cluster peers

    const T* __restrict__ gamma = static_cast<const T*>(a.gamma);
    const T* __restrict__ beta = static_cast<const T*>(a.beta);
    const int T_ = blockDim.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T_ >> 5;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int64_t first_row = blockIdx.x / C;
    const int64_t row_step = gridDim.x / C;
    const int nacc = (a.N + VEC - 1) / VEC;
    const int rounds = a.rounds;

    int buf = 0;
    for (int64_t row = first_row; row < a.M; row += row_step, buf ^= 1) {
        const T* xr = static_cast<const T*>(a.x) + row * a.N;
        T* yr = static_cast<T*>(a.y) + row * a.N;

        Frag<T, VEC> f[V];
        bool ok[V];
        Welford st = welford_empty();
        float ss = 0.f;
        float K = 0.f;
        if constexpr (LN) {
            Frag<T, 1> k0;
            k0.load(xr);
            K = k0.get(0);
        }
        for (int r = 0; r < rounds; ++r) {
            const int base = (r * static_cast<int>(C) + static_cast<int>(rank)) * V * T_ + tid;
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int acc = base + j * T_;
                ok[j] = acc < nacc;
                if (ok[j]) f[j].load(xr + acc * VEC);
            }
            if constexpr (LN)
                st = chan_merge(st, thread_welford<T, VEC, V>(f, ok, K));
            else
                ss += thread_sumsq<T, VEC, V>(f, ok);
        }

        // warps -> shared memory -> every warp merges the per-warp states
        float mu = 0.f, rs;
        if constexpr (LN) {
            st = group_merge(st, 32);
            if (lane == 0) {
                warp_part[buf][0][warp] = st.n;
                warp_part[buf][1][warp] = st.mean;
                warp_part[buf][2][warp] = st.m2;
            }
            __syncthreads();
            st = lane < nwarps ? Welford{warp_part[buf][0][lane], warp_part[buf][1][lane], warp_part[buf][2][lane]}
                               : welford_empty();
            st = group_merge(st, 32);
            if (C > 1) {
                if (tid == 0) {
                    cta_part[buf][0] = st.n;
                    cta_part[buf][1] = st.mean;
                    cta_part[buf][2] = st.m2;
                }
                cluster_barrier();
                Welford p = welford_empty();
                if (lane < static_cast<int>(C)) {
                    p.n = ld_peer_f32(peer_smem_addr(&cta_part[buf][0], lane));
                    p.mean = ld_peer_f32(peer_smem_addr(&cta_part[buf][1], lane));
                    p.m2 = ld_peer_f32(peer_smem_addr(&cta_part[buf][2], lane));
                }
                st = group_merge(p, 32);
            }
            mu = st.mean;
            rs = rsqrtf(st.m2 / static_cast<float>(a.N) + a.eps);
            if (rank == 0 && tid == 0) {
                if (a.mean) a.mean[row] = K + mu;
                if (a.rstd) a.rstd[row] = rs;
            }
        } else {
            ss = group_sum(ss, 32);
            if (lane == 0) warp_part[buf][0][warp] = ss;
            __syncthreads();
            ss = group_sum(lane < nwarps ? warp_part[buf][0][lane] : 0.f, 32);
            if (C > 1) {
                if (tid == 0) cta_part[buf][0] = ss;
                cluster_barrier();
                ss = group_sum(lane < static_cast<int>(C) ? ld_peer_f32(peer_smem_addr(&cta_part[buf][0], lane)) : 0.f,
                               32);
            }
            rs = rsqrtf(ss / static_cast<float>(a.N) + a.eps);
        }

        for (int r = rounds - 1; r >= 0; --r) {
            const int base = (r * static_cast<int>(C) + static_cast<int>(rank)) * V * T_ + tid;
            if (r != rounds - 1) {
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const int acc = base + j * T_;
                    ok[j] = acc < nacc;
                    if (ok[j]) f[j].load(xr + acc * VEC);
                }
            }
#pragma unroll
            for (int j = 0; j < V; ++j)
                if (ok[j]) emit<T, VEC, LN>(f[j], gamma, beta, yr, (base + j * T_) * VEC, K, mu, rs);
        }
    }
    // No CTA may exit while a peer can still read its shared memory.
    if (C > 1) cluster_barrier();
}

// ----------------------------------------------------------------- launch
template <class T, bool LN>
using KernelFn = void (*)(const NormArgs);

template <class T, bool LN, int VEC>
KernelFn<T, LN> pick_kernel(int mapping, int per_thread) {
    const bool group = mapping == NORM_MAP_GROUP;
    switch (per_thread) {
        case 1: return group ? norm_fwd_group<T, VEC, 1, LN> : norm_fwd_cta<T, VEC, 1, LN>;
        case 2: return group ? norm_fwd_group<T, VEC, 2, LN> : norm_fwd_cta<T, VEC, 2, LN>;
        case 4: return group ? norm_fwd_group<T, VEC, 4, LN> : norm_fwd_cta<T, VEC, 4, LN>;
        case 8: return group ? norm_fwd_group<T, VEC, 8, LN> : norm_fwd_cta<T, VEC, 8, LN>;
        default: return nullptr;
    }
}

template <class T, bool LN>
cudaError_t launch_norm(const norm_plan& p, const NormArgs& a, cudaStream_t stream) {
    KernelFn<T, LN> k = p.vec_elems == 1 ? pick_kernel<T, LN, 1>(p.mapping, p.per_thread)
                                         : pick_kernel<T, LN, ElemVec<T>::value>(p.mapping, p.per_thread);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.mapping == NORM_MAP_CTA && p.cluster > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace libnorm
