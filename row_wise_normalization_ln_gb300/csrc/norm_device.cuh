// Device building blocks of the row-wise LayerNorm / RMSNorm forward kernels:
// the Welford state and its parallel merge, warp butterflies, cluster
// (distributed shared memory) primitives, and 128-bit / element accesses.
//
// Sources (page title, section):
//   [Ch7] "第 7 章 LayerNorm 与 RMSNorm": §7.4 Welford state (n, mean, M2),
//         §7.4.1 parallel merge, §7.4.2 warp xor-shuffle reduction,
//         §7.6 two-level (warp, then shared memory) block reduction.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace libnorm {

constexpr unsigned kFullMask = 0xffffffffu;

// ----------------------------------------------------------------- Welford
// (n, mean, M2) of a set of elements ([Ch7] §7.4). The count is a float:
// every count here is an integer <= 2^24, which fp32 holds exactly.
struct Welford {
    float n, mean, m2;
};

__device__ __forceinline__ Welford welford_empty() { return {0.f, 0.f, 0.f}; }

// Parallel merge ([Ch7] §7.4.1): n = na+nb, d = mb-ma, mean = ma + d*nb/n,
// M2 = M2a + M2b + d^2*na*nb/n. Merging with an empty state returns the other
// state exactly; two empty states give an empty state.
__device__ __forceinline__ Welford chan_merge(const Welford& a, const Welford& b) {
    const float n = a.n + b.n;
    if (n == 0.f) return welford_empty();
    const float wb = b.n / n;
    const float d = b.mean - a.mean;
    Welford r;
    r.n = n;
    r.mean = fmaf(d, wb, a.mean);
    r.m2 = a.m2 + b.m2 + d * d * a.n * wb;
    return r;
}

__device__ __forceinline__ Welford shfl_xor(const Welford& s, int off) {
    Welford o;
    o.n = __shfl_xor_sync(kFullMask, s.n, off);
    o.mean = __shfl_xor_sync(kFullMask, s.mean, off);
    o.m2 = __shfl_xor_sync(kFullMask, s.m2, off);
    return o;
}

// Xor butterfly over aligned groups of `width` lanes (a power of two <= 32;
// every lane of the warp must call it). The merge is not bitwise symmetric,
// so the lower lane's state is always the left operand: both lanes of a pair
// compute the identical merge and every lane of the group ends with
// bit-identical statistics.
__device__ __forceinline__ Welford group_merge(Welford s, int width) {
    const int lane = threadIdx.x & 31;
    for (int off = width >> 1; off > 0; off >>= 1) {
        const Welford o = shfl_xor(s, off);
        s = (lane & off) ? chan_merge(o, s) : chan_merge(s, o);
    }
    return s;
}

// Sum butterfly (RMSNorm's sum of squares); fp32 addition is commutative, so
// every lane of the group ends with the same bits.
__device__ __forceinline__ float group_sum(float v, int width) {
    for (int off = width >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
    return v;
}

// ----------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives; shared-memory writes
// made before the barrier are visible to cluster peers after it. This is a
// hardware barrier (no polling loop): it completes once all CTAs of the
// cluster, which are co-scheduled, have arrived.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Address of `p` (a __shared__ variable of this CTA) in the shared memory
// window of cluster peer `rank`.
__device__ __forceinline__ uint32_t peer_smem_addr(const void* p, uint32_t rank) {
    const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}

__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ----------------------------------------------------------------- accesses
// One global access of VEC consecutive elements: a 16-byte vector (4 fp32 or
// 8 bf16) when the row allows it, otherwise a single element. bf16 values are
// widened exactly (the bf16 pattern is the top half of the fp32 pattern).
template <class T, int VEC>
struct Frag;

template <>
struct Frag<float, 4> {
    float4 v;
    __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
    __device__ __forceinline__ void load_param(const float* p) { v = __ldg(reinterpret_cast<const float4*>(p)); }
    __device__ __forceinline__ float get(int e) const {
        return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&o)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
    }
};

template <>
struct Frag<__nv_bfloat16, 8> {
    uint4 v;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint4*>(p); }
    __device__ __forceinline__ void load_param(const __nv_bfloat16* p) { v = __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ __forceinline__ float get(int e) const {
        const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
        return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // round to nearest-even
        return *reinterpret_cast<const uint32_t*>(&b);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&o)[8]) {
        uint4 w;
        w.x = pack(o[0], o[1]);
        w.y = pack(o[2], o[3]);
        w.z = pack(o[4], o[5]);
        w.w = pack(o[6], o[7]);
        *reinterpret_cast<uint4*>(p) = w;
    }
};

template <>
struct Frag<float, 1> {
    float v;
    __device__ __forceinline__ void load(const float* p) { v = *p; }
    __device__ __forceinline__ void load_param(const float* p) { v = __ldg(p); }
    __device__ __forceinline__ float get(int) const { return v; }
    static __device__ __forceinline__ void store(float* p, const float (&o)[1]) { *p = o[0]; }
};

template <>
struct Frag<__nv_bfloat16, 1> {
    uint32_t v;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        v = *reinterpret_cast<const unsigned short*>(p);
    }
    __device__ __forceinline__ void load_param(const __nv_bfloat16* p) {
        v = __ldg(reinterpret_cast<const unsigned short*>(p));
    }
    __device__ __forceinline__ float get(int) const { return __uint_as_float(v << 16); }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&o)[1]) {
        *p = __float2bfloat16_rn(o[0]);
    }
};

}  // namespace libnorm
