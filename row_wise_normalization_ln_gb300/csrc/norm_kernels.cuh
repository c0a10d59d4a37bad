// Row-wise LayerNorm / RMSNorm forward kernels for sm_103a.
//
// Every kernel reads x from HBM once, keeps its slice of the row in
// registers, reduces the statistics in fp32 and writes y in the same pass
// (fused affine and cast):
//
//   norm_fwd_group  `group` lanes of a warp own a row (short rows).
//   norm_fwd_cta    a CTA, or a thread-block cluster, owns a row; rows longer
//                   than one pass of the cluster's registers are walked in
//                   rounds. Also the element-access path for unaligned rows.
//   norm_fwd_ring   the CTA mapping on a persistent grid: bulk copies bring
//                   each CTA's share of its next rows into a shared-memory
//                   ring while it works on the current one, and each thread
//                   widens its elements to fp32 once.
//
// Inside a CTA's slice the layout is warp-major: warp w holds V runs of 32
// consecutive accesses, access (w*V + j)*32 + lane, so every instruction
// touches 32 consecutive accesses and the offset of run j is a compile-time
// constant.
//
// LayerNorm statistics ([Ch7] §7.4, §7.4.1): each thread forms the Welford
// state (n_t, mean_t, M2_t) of its own elements, shifted by the row's first
// element K, by two passes over its registers ([T3] §② trap 2: the row is
// in registers, so "two passes" cost no memory traffic); on 16-bit rows, by
// two passes over each 16-byte access and the pairwise merge of the access
// states (Slice::welford). The states of all
// threads of the row are then merged with the merge rule in its k-way form,
//     mean = sum_t n_t mean_t / N,    M2 = sum_t (M2_t + n_t (mean_t - mean)^2),
// which is what any sequence of pairwise merges reaches; each sum is an xor
// butterfly inside the warp, then shared memory across warps, then
// distributed shared memory across the cluster. The variance is never formed
// as E[x^2] - E[x]^2. Elements beyond N are never loaded and never counted
// ([T3] §② trap 1). The shift keeps the digits of rows whose mean dwarfs
// their spread ([Ch7] §7.3): x - K of nearby values is exact and the merged
// means stay small.
//
// Sources (page title, section):
//   [Ch7] "第 7 章 LayerNorm 与 RMSNorm": §7.1, §7.3-7.6.
//   [T3]  "T3 讲解：LayerNorm / RMSNorm 的 forward": §②, §③.
#pragma once

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "norm_args.h"
#include "norm_device.cuh"

namespace libnorm {

template <class T>
struct ElemVec {
    static constexpr int value = 16 / sizeof(T);
};

// ================================================================== element math
// One access is a 16-byte vector (4 fp32, or 8 bf16 or fp16) held as a
// uint4, or a single element (VEC = 1) held in the low bits of a uint32.
// 16-bit values are widened exactly (a bf16 pattern is the top half of an
// fp32 pattern; every fp16 value is an fp32 value).

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // round to nearest-even
    return *reinterpret_cast<const uint32_t*>(&b);
}

// bf16 rows widen each pair of values exactly to an fp32 pair and work on it
// with the sm_100-family packed instructions (two IEEE fp32 operations, each
// rounded to nearest-even, per instruction); fp32 rows use scalar fp32
// instructions (measured faster there).
__device__ __forceinline__ float2 f2_splat(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 bf16x2_widen(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

// A pair of 16-bit values in one 32-bit word: exact widening to an fp32
// pair, and nearest-even rounding of an fp32 pair back.
struct Bf16Pair {
    static __device__ __forceinline__ float2 widen(uint32_t w) { return bf16x2_widen(w); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16x2(lo, hi); }
    // (lo + c, hi + c) in fp32, each widened exactly and rounded once. For
    // bf16 the widening is a shift and a mask and one packed add follows
    // (the mixed-precision add measured more instructions here).
    static __device__ __forceinline__ float2 add(uint32_t w, float c) { return __fadd2_rn(widen(w), f2_splat(c)); }
};
struct F16Pair {
    static __device__ __forceinline__ float2 widen(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));  // every fp16 value is an fp32 value
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        const __half2 h = __floats2half2_rn(lo, hi);  // round to nearest-even
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    // The same for fp16 with the sm_100-family mixed-precision add, which
    // takes the 16-bit halves directly (measured faster than converting
    // the pair and adding).
    static __device__ __forceinline__ float2 add(uint32_t w, float c) {
        float2 r;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.f16 %0, l, %3;\n\tadd.rn.f32.f16 %1, h, %3;\n\t}"
            : "=f"(r.x), "=f"(r.y)
            : "r"(w), "f"(c));
        return r;
    }
};

// 16-byte global loads with an L1 allocation hint, for data a thread reads
// once: `stream` does not allocate the line in L1 and, as volatile asm with
// a memory clobber, stays after this thread's earlier stores (it may read
// a line the thread wrote); `first` allocates the line first in line for
// eviction and is for data this kernel has not written before the load
// (the compiler may move it like any pure computation). Both read through
// the coherent path. Each use states the measurement it rests on.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_first_v4(const void* p) {
    uint4 v;
    asm("ld.global.L1::evict_first.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Per-access operations, specialised on element type and width.
template <class T, int VEC>
struct Ops;

template <>
struct Ops<float, 4> {
    using Raw = uint4;
    static __device__ __forceinline__ float e(const Raw& r, int i) {
        return __uint_as_float(i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w);
    }
    // sum of (x - K)
    static __device__ __forceinline__ float shifted_sum(const Raw& r, float K) {
        return ((e(r, 0) - K) + (e(r, 1) - K)) + ((e(r, 2) - K) + (e(r, 3) - K));
    }
    // acc + sum ((x - K) - mu)^2
    static __device__ __forceinline__ float dev2(const Raw& r, float K, float mu, float acc) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float d = (e(r, i) - K) - mu;
            acc = fmaf(d, d, acc);
        }
        return acc;
    }
    static __device__ __forceinline__ float sumsq(const Raw& r, float acc) {
#pragma unroll
        for (int i = 0; i < 4; ++i) acc = fmaf(e(r, i), e(r, i), acc);
        return acc;
    }
    // LayerNorm: ((x - K) * rs + nmr) * gamma + beta with nmr = -mu * rs
    static __device__ __forceinline__ Raw ln_out(const Raw& r, float K, float rs, float nmr, const Raw& g,
                                                 const Raw& b) {
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = fmaf(fmaf(e(r, i) - K, rs, nmr), e(g, i), e(b, i));
        return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                          __float_as_uint(o[3]));
    }
    // RMSNorm: (x * w) * rs
    static __device__ __forceinline__ Raw rms_out(const Raw& r, float rs, const Raw& w) {
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = (e(r, i) * e(w, i)) * rs;
        return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                          __float_as_uint(o[3]));
    }
    // The same fp32 values, unrounded (for a quantised output).
    static __device__ __forceinline__ void ln_vals(const Raw& r, float K, float rs, float nmr, const Raw& g,
                                                   const Raw& b, float* o) {
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = fmaf(fmaf(e(r, i) - K, rs, nmr), e(g, i), e(b, i));
    }
    static __device__ __forceinline__ void rms_vals(const Raw& r, float rs, const Raw& w, float* o) {
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = (e(r, i) * e(w, i)) * rs;
    }
    // Residual add h = x + r, each element rounded once to fp32.
    static __device__ __forceinline__ Raw add_round(const Raw& x, const Raw& r) {
        return make_uint4(__float_as_uint(e(x, 0) + e(r, 0)), __float_as_uint(e(x, 1) + e(r, 1)),
                          __float_as_uint(e(x, 2) + e(r, 2)), __float_as_uint(e(x, 3) + e(r, 3)));
    }
    static __device__ __forceinline__ Raw load(const float* p) { return *reinterpret_cast<const uint4*>(p); }
    static __device__ __forceinline__ Raw load_stream(const float* p) { return ld_stream_v4(p); }
    static __device__ __forceinline__ Raw load_first(const float* p) { return ld_first_v4(p); }
    static __device__ __forceinline__ Raw load_param(const float* p) {
        return __ldg(reinterpret_cast<const uint4*>(p));
    }
    // The same access assembled from element loads (p not 16-byte aligned).
    static __device__ __forceinline__ Raw load_param_elems(const float* p) {
        return make_uint4(__float_as_uint(__ldg(p)), __float_as_uint(__ldg(p + 1)), __float_as_uint(__ldg(p + 2)),
                          __float_as_uint(__ldg(p + 3)));
    }
    static __device__ __forceinline__ void store(float* p, const Raw& v) { *reinterpret_cast<uint4*>(p) = v; }
};

// Eight 16-bit elements (bf16 or fp16) per access, worked on as fp32 pairs.
template <class T, class P>
struct Ops16 {
    using Raw = uint4;
    static __device__ __forceinline__ uint32_t w(const Raw& r, int i) {
        return i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w;
    }
    // x - K of a word's two elements (exact widening, one rounding).
    static __device__ __forceinline__ float2 shifted(uint32_t wd, float K) { return P::add(wd, -K); }
    static __device__ __forceinline__ float shifted_sum(const Raw& r, float K) {
        const float2 a = __fadd2_rn(shifted(r.x, K), shifted(r.y, K));
        const float2 b = __fadd2_rn(shifted(r.z, K), shifted(r.w, K));
        const float2 s = __fadd2_rn(a, b);
        return s.x + s.y;
    }
    static __device__ __forceinline__ float dev2(const Raw& r, float K, float mu, float acc) {
        const float2 nm = f2_splat(-mu);
        float2 q = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 d = __fadd2_rn(shifted(w(r, i), K), nm);
            q = __ffma2_rn(d, d, q);
        }
        return acc + (q.x + q.y);
    }
    static __device__ __forceinline__ float sumsq(const Raw& r, float acc) {
        float2 q = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = P::widen(w(r, i));
            q = __ffma2_rn(x, x, q);
        }
        return acc + (q.x + q.y);
    }
    static __device__ __forceinline__ Raw ln_out(const Raw& r, float K, float rs, float nmr, const Raw& g,
                                                 const Raw& b) {
        const float2 rs2 = f2_splat(rs), nm2 = f2_splat(nmr);
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 y = __ffma2_rn(__ffma2_rn(shifted(w(r, i), K), rs2, nm2), P::widen(w(g, i)), P::widen(w(b, i)));
            o[i] = P::pack(y.x, y.y);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
    static __device__ __forceinline__ Raw rms_out(const Raw& r, float rs, const Raw& wt) {
        const float2 rs2 = f2_splat(rs);
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 y = __fmul2_rn(__fmul2_rn(P::widen(w(r, i)), P::widen(w(wt, i))), rs2);
            o[i] = P::pack(y.x, y.y);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
    static __device__ __forceinline__ void ln_vals(const Raw& r, float K, float rs, float nmr, const Raw& g,
                                                   const Raw& b, float* o) {
        const float2 rs2 = f2_splat(rs), nm2 = f2_splat(nmr);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 y = __ffma2_rn(__ffma2_rn(shifted(w(r, i), K), rs2, nm2), P::widen(w(g, i)), P::widen(w(b, i)));
            o[2 * i] = y.x;
            o[2 * i + 1] = y.y;
        }
    }
    static __device__ __forceinline__ void rms_vals(const Raw& r, float rs, const Raw& wt, float* o) {
        const float2 rs2 = f2_splat(rs);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 y = __fmul2_rn(__fmul2_rn(P::widen(w(r, i)), P::widen(w(wt, i))), rs2);
            o[2 * i] = y.x;
            o[2 * i + 1] = y.y;
        }
    }
    // Residual add h = x + r: fp32 carries at least 2p + 2 bits for both
    // 16-bit formats (p = 8 for bf16, 11 for fp16), so rounding the fp32 sum
    // to T rounds the exact sum once.
    static __device__ __forceinline__ Raw add_round(const Raw& x, const Raw& r) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 h = __fadd2_rn(P::widen(w(x, i)), P::widen(w(r, i)));
            o[i] = P::pack(h.x, h.y);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
    static __device__ __forceinline__ Raw load(const T* p) { return *reinterpret_cast<const uint4*>(p); }
    static __device__ __forceinline__ Raw load_stream(const T* p) { return ld_stream_v4(p); }
    static __device__ __forceinline__ Raw load_first(const T* p) { return ld_first_v4(p); }
    static __device__ __forceinline__ Raw load_param(const T* p) {
        return __ldg(reinterpret_cast<const uint4*>(p));
    }
    static __device__ __forceinline__ Raw load_param_elems(const T* p) {
        const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = static_cast<uint32_t>(__ldg(q + 2 * i)) | (static_cast<uint32_t>(__ldg(q + 2 * i + 1)) << 16);
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
    static __device__ __forceinline__ void store(T* p, const Raw& v) {
        *reinterpret_cast<uint4*>(p) = v;
    }
};

template <>
struct Ops<__nv_bfloat16, 8> : Ops16<__nv_bfloat16, Bf16Pair> {};
template <>
struct Ops<__half, 8> : Ops16<__half, F16Pair> {};

// Single elements (rows that are not whole 16-byte aligned vectors).
template <class T>
struct ScalarOps {
    using Raw = uint32_t;
    static __device__ __forceinline__ float e(Raw r) {
        if constexpr (sizeof(T) == 4)
            return __uint_as_float(r);
        else if constexpr (std::is_same<T, __half>::value)
            return __half2float(__ushort_as_half(static_cast<unsigned short>(r)));
        else
            return __uint_as_float(r << 16);
    }
    static __device__ __forceinline__ float shifted_sum(Raw r, float K) { return e(r) - K; }
    static __device__ __forceinline__ float dev2(Raw r, float K, float mu, float acc) {
        const float d = (e(r) - K) - mu;
        return fmaf(d, d, acc);
    }
    static __device__ __forceinline__ float sumsq(Raw r, float acc) { return fmaf(e(r), e(r), acc); }
    static __device__ __forceinline__ Raw ln_out(Raw r, float K, float rs, float nmr, Raw g, Raw b) {
        return from_float(fmaf(fmaf(e(r) - K, rs, nmr), e(g), e(b)));
    }
    static __device__ __forceinline__ Raw rms_out(Raw r, float rs, Raw wt) { return from_float((e(r) * e(wt)) * rs); }
    static __device__ __forceinline__ void ln_vals(Raw r, float K, float rs, float nmr, Raw g, Raw b, float* o) {
        o[0] = fmaf(fmaf(e(r) - K, rs, nmr), e(g), e(b));
    }
    static __device__ __forceinline__ void rms_vals(Raw r, float rs, Raw wt, float* o) { o[0] = (e(r) * e(wt)) * rs; }
    static __device__ __forceinline__ Raw add_round(Raw x, Raw r) { return from_float(e(x) + e(r)); }
    static __device__ __forceinline__ Raw from_float(float v) {
        if constexpr (sizeof(T) == 4)
            return __float_as_uint(v);
        else if constexpr (std::is_same<T, __half>::value)
            return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v)));
        else
            return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
    }
    static __device__ __forceinline__ Raw load(const T* p) {
        if constexpr (sizeof(T) == 4)
            return __float_as_uint(*reinterpret_cast<const float*>(p));
        else
            return *reinterpret_cast<const unsigned short*>(p);
    }
    static __device__ __forceinline__ Raw load_param(const T* p) {
        if constexpr (sizeof(T) == 4)
            return __float_as_uint(__ldg(reinterpret_cast<const float*>(p)));
        else
            return __ldg(reinterpret_cast<const unsigned short*>(p));
    }
    static __device__ __forceinline__ Raw load_param_elems(const T* p) { return load_param(p); }
    // Element accesses take no L1 hint.
    static __device__ __forceinline__ Raw load_stream(const T* p) { return load(p); }
    static __device__ __forceinline__ Raw load_first(const T* p) { return load(p); }
    static __device__ __forceinline__ void store(T* p, Raw v) {
        if constexpr (sizeof(T) == 4)
            *reinterpret_cast<float*>(p) = __uint_as_float(v);
        else
            *reinterpret_cast<unsigned short*>(p) = static_cast<unsigned short>(v);
    }
};

template <class T, int VEC>
using OpsFor = typename std::conditional<VEC == 1, ScalarOps<T>, Ops<T, VEC>>::type;

// The row's first element, the shift K of LayerNorm; with a residual, the
// first element of h = x + r (rounded as the stored h is).
template <class T>
__device__ __forceinline__ float first_elem(const T* row) {
    return ScalarOps<T>::e(ScalarOps<T>::load(row));
}
template <class T>
__device__ __forceinline__ float first_elem_add(const T* xrow, const T* rrow) {
    using SO = ScalarOps<T>;
    return SO::e(SO::add_round(SO::load(xrow), SO::load(rrow)));
}

// FP8 output ([Ch7] §7.9: the norm writes the next GEMM's quantised input):
// VEC fp32 values times the inverse of the static scale, converted to OCP
// FP8 E4M3 with the hardware's round-to-nearest-even, saturating conversion
// (magnitudes from 448 give +-448), stored as VEC bytes.
template <int VEC>
__device__ __forceinline__ void store_e4m3(uint8_t* p, const float* o, float inv) {
    if constexpr (VEC == 1) {
        *p = static_cast<uint8_t>(__nv_cvt_float_to_fp8(o[0] * inv, __NV_SATFINITE, __NV_E4M3));
    } else {
        uint32_t q[VEC / 4];
#pragma unroll
        for (int k = 0; k < VEC / 4; ++k) {
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(o[4 * k] * inv, o[4 * k + 1] * inv),
                                                         __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(o[4 * k + 2] * inv, o[4 * k + 3] * inv),
                                                         __NV_SATFINITE, __NV_E4M3);
            q[k] = lo | (hi << 16);
        }
        if constexpr (VEC == 4)
            *reinterpret_cast<uint32_t*>(p) = q[0];
        else
            *reinterpret_cast<uint2*>(p) = make_uint2(q[0], q[1]);
    }
}

// ================================================================== a thread's slice
// V accesses of one row held in registers as loaded; the first `nvalid` lie
// inside the row. `stride` is the distance in elements between a thread's
// consecutive accesses (32*VEC in the warp-major CTA layout, G*VEC in the
// GROUP layout). LayerNorm works on x - K (K set by set_shift).
template <class T, int VEC, int V, bool LN>
struct Slice {
    using O = OpsFor<T, VEC>;
    typename O::Raw raw[V];
    float K;

    __device__ __forceinline__ void set_shift(float k) { K = k; }
    __device__ __forceinline__ void set(int j, const typename O::Raw& v) { raw[j] = v; }
    // HINT: the loads do not allocate in L1 (O::load_stream).
    template <bool HINT = false>
    __device__ __forceinline__ void load(const T* p, int stride, int nvalid) {
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) raw[j] = HINT ? O::load_stream(p + j * stride) : O::load(p + j * stride);
    }
    // Fused residual add: hold h = x + r (rounded to T). h is stored later,
    // by store_h, once every thread of the row has read its inputs (h may be
    // the x or r buffer itself). HINT: x and r evict first from L1.
    template <bool HINT = false>
    __device__ __forceinline__ void load_add(const T* px, const T* pr, int stride, int nvalid) {
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid)
                raw[j] = HINT ? O::add_round(O::load_first(px + j * stride), O::load_first(pr + j * stride))
                              : O::add_round(O::load(px + j * stride), O::load(pr + j * stride));
    }
    __device__ __forceinline__ void store_h(T* ph, int stride, int nvalid) const {
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) O::store(ph + j * stride, raw[j]);
    }
    // Welford state of the valid elements. 16-bit rows: each access's eight
    // values of x - K get their own two-pass state (sum, mean, M2 about
    // that mean) and are merged into the thread's running state with the
    // pairwise merge rule ([Ch7] §7.4.1); after j accesses the thread holds
    // 8j values, so the weights 1/(j+1) and 8j/(j+1) are constants. This
    // widens each value once for the statistics. Other rows: two passes
    // over the registers, the sum and mean of x - K, then M2 about that mean.
    // STREAM selects the per-access form for 16-bit rows (the fused-add
    // kernels measured slower with it, and the cluster kernels, which no
    // benchmark shape measured, keep the two passes too).
    template <bool STREAM = true>
    __device__ __forceinline__ void welford(int nvalid, float inv_n, float& sum, float& mean, float& m2) const {
        if constexpr (VEC == 8 && STREAM) {
            float sum_r = 0.f, mean_r = 0.f, m2_r = 0.f;
#pragma unroll
            for (int j = 0; j < V; ++j)
                if (j < nvalid) {
                    float2 d[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) d[i] = O::shifted(O::w(raw[j], i), K);
                    const float2 t = __fadd2_rn(__fadd2_rn(d[0], d[1]), __fadd2_rn(d[2], d[3]));
                    const float sj = t.x + t.y;
                    const float mj = sj * 0.125f;
                    const float2 nm = f2_splat(-mj);
                    float2 q = make_float2(0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 e = __fadd2_rn(d[i], nm);
                        q = __ffma2_rn(e, e, q);
                    }
                    const float qj = q.x + q.y;
                    if (j == 0) {
                        mean_r = mj;
                        m2_r = qj;
                    } else {
                        const float dm = mj - mean_r;
                        mean_r = fmaf(dm, 1.f / static_cast<float>(j + 1), mean_r);
                        m2_r = fmaf(dm * dm, 8.f * static_cast<float>(j) / static_cast<float>(j + 1), m2_r + qj);
                    }
                    sum_r += sj;
                }
            sum = sum_r;
            mean = mean_r;
            m2 = m2_r;
            return;
        }
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
                if (j & 1)
                    s1 += O::shifted_sum(raw[j], K);
                else
                    s0 += O::shifted_sum(raw[j], K);
            }
        sum = s0 + s1;
        mean = sum * inv_n;
        float q0 = 0.f, q1 = 0.f;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
                if (j & 1)
                    q1 = O::dev2(raw[j], K, mean, q1);
                else
                    q0 = O::dev2(raw[j], K, mean, q0);
            }
        m2 = q0 + q1;
    }
    // Sum of squares of the valid elements (RMSNorm, [Ch7] §7.5.1).
    __device__ __forceinline__ float sumsq(int nvalid) const {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
                if (j & 1)
                    s1 = O::sumsq(raw[j], s1);
                else
                    s0 = O::sumsq(raw[j], s0);
            }
        return s0 + s1;
    }
    // Normalise, apply the affine parameters, round and store the valid
    // accesses; `g`, `b` and `y` point at this thread's first access.
    // LayerNorm: y = ((x - K) * rstd - mu * rstd) * gamma + beta, where mu is
    // the mean of x - K (so x - mean is never formed from a rounded fp32
    // mean); RMSNorm: y = (x * w) * rstd.
    // gamma/beta access j, as one vector load, or element by element when
    // `sp` (their vectors are not 16-byte aligned in this row).
    static __device__ __forceinline__ typename O::Raw param(const T* p, bool sp) {
        return sp ? O::load_param_elems(p) : O::load_param(p);
    }
    __device__ __forceinline__ void emit(const T* g, const T* b, T* y, int stride, int nvalid, float mu, float rs,
                                         bool sp = false) const {
        const float nmr = -mu * rs;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
                if constexpr (LN)
                    O::store(y + j * stride, O::ln_out(raw[j], K, rs, nmr, param(g + j * stride, sp),
                                                       param(b + j * stride, sp)));
                else
                    O::store(y + j * stride, O::rms_out(raw[j], rs, param(g + j * stride, sp)));
            }
    }
    // emit with an FP8 E4M3 output: the same fp32 values, scaled by `inv`
    // (1 / the static scale) and quantised; `y8` points at this thread's
    // first access in bytes (one byte per element).
    __device__ __forceinline__ void emit_q8(const T* g, const T* b, uint8_t* y8, int stride, int nvalid, float mu,
                                            float rs, float inv, bool sp = false) const {
        const float nmr = -mu * rs;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
                float o[VEC];
                if constexpr (LN)
                    O::ln_vals(raw[j], K, rs, nmr, param(g + j * stride, sp), param(b + j * stride, sp), o);
                else
                    O::rms_vals(raw[j], rs, param(g + j * stride, sp), o);
                store_e4m3<VEC>(y8 + j * stride, o, inv);
            }
    }
    // Output step of either kind.
    template <bool Q8>
    __device__ __forceinline__ void out(const T* g, const T* b, void* y, int64_t offset, int stride, int nvalid,
                                        float mu, float rs, float inv, bool sp = false) const {
        if constexpr (Q8)
            emit_q8(g, b, static_cast<uint8_t*>(y) + offset, stride, nvalid, mu, rs, inv, sp);
        else
            emit(g, b, static_cast<T*>(y) + offset, stride, nvalid, mu, rs, sp);
    }
};

// How many of a thread's V runs lie inside a row of `nacc` accesses when its
// first access is `first` and its runs are `stride_acc` accesses apart.
__device__ __forceinline__ int valid_runs(int nacc, int first, int stride_acc, int V) {
    if (first >= nacc) return 0;
    return min(V, (nacc - first + stride_acc - 1) / stride_acc);
}

// ================================================================== row reduction
// Sum of one value per thread over the CTA and, when C > 1, over the
// cluster: xor butterfly in each warp, per-warp partials in shared memory, a
// butterfly over them in every warp, then the CTAs' partials over
// distributed shared memory. Every thread of every CTA of the cluster
// returns the same bits.
//
// A row makes two such sums for LayerNorm (stage 0, then stage 1), so a
// slot is written again only after a barrier that every reader of its
// previous value has passed. RMSNorm makes one, in the stage its caller
// names: kernels that walk several rows per CTA either alternate the stage
// from row to row or put a barrier between rows.
struct RowReduceSmem {
    float warp_part[2][32];   // [stage][warp]
    float cta_part[2];        // [stage], read by cluster peers
    static constexpr bool kWarpStates = false;
    float2 warp_pair[32];     // [warp]: LayerNorm in a cluster, (sum, count) of each warp
    float cta_state[2][4];    // [stage]: LayerNorm in a cluster, (count, sum, M2) of this CTA, read by peers
};

// Kernels launched with clusters: also each warp's LayerNorm state
// (count, sum, M2, -), read by peers when the cluster has at most 32 warps.
struct RowReduceSmemCl : RowReduceSmem {
    static constexpr bool kWarpStates = true;
    float4 warp_state[2][32];  // [stage][warp]
};

// Sums of a pair per thread over the CTA (no cluster): butterflies in each
// warp, per-warp pairs in shared memory, butterflies over them in every
// warp. Uses the slots of stage 0.
__device__ __forceinline__ float2 cta_sum2(RowReduceSmem& red, float a, float b, int nwarps, int wwidth) {
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    a = group_sum(a, 32);
    b = group_sum(b, 32);
    if (lane == 0) red.warp_pair[tid >> 5] = make_float2(a, b);
    __syncthreads();
    const float2 w = lane < nwarps ? red.warp_pair[lane] : make_float2(0.f, 0.f);
    return make_float2(sum_first_lanes(w.x, wwidth), sum_first_lanes(w.y, wwidth));
}

template <bool EARLY = false>
__device__ __forceinline__ float row_sum(RowReduceSmem& red, int stage, float v, uint32_t C, int nwarps,
                                         int wwidth) {
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    v = group_sum(v, 32);
    if (lane == 0) red.warp_part[stage][tid >> 5] = v;
    __syncthreads();
    v = sum_first_lanes(lane < nwarps ? red.warp_part[stage][lane] : 0.f, wwidth);
    if (C > 1) {
        if (tid == 0) red.cta_part[stage] = v;
        cluster_barrier();
        v = sum_first_lanes(
            lane < static_cast<int>(C) ? ld_peer_f32(peer_smem_addr(&red.cta_part[stage], lane)) : 0.f,
            static_cast<int>(C));
        if constexpr (EARLY) cluster_arrive();  // done with the peers' slots; the caller waits
    }
    return v;
}

// Row statistics from each thread's Welford state (LayerNorm) or sum of
// squares (RMSNorm): the shifted mean mu and rstd, identical in every thread
// of every CTA of the cluster. LayerNorm, one CTA per row: the k-way merge
// of the threads' states, two sums. LayerNorm over a cluster, one cluster
// barrier per row: with at most 32 warps in the cluster (every default
// plan), each warp merges its lanes' states and publishes its own, and every
// warp merges all the cluster's warp states after the exchange; with more,
// each CTA first merges its threads' states into its own (n_c, mean_c,
// M2_c) and every thread merges the C CTA states in rank order. Both use
// the merge rule of [Ch7] §7.4.1 in its k-way form. `stage`: the stage of
// RMSNorm's one sum, and of the states a LayerNorm cluster publishes
// (callers that walk several rows per CTA alternate it or put a barrier
// between rows).
// EARLY (C > 1 only): each thread arrives at the next cluster barrier as
// soon as it has read the peers' values, and the caller waits on it before
// this CTA's slot is written again or the CTA exits, so that the wait
// costs nothing once the peers are past their own reads (a full barrier
// there would wait for the slowest peer's whole output pass).
template <bool LN, bool EARLY = false, class Red>
__device__ __forceinline__ void row_stats(Red& red, float n_t, float sum_t, float mean_t, float m2_t,
                                          float ss_t, float invN, float eps, uint32_t C, int nwarps, int wwidth,
                                          int stage, float& mu, float& rs) {
    if constexpr (LN) {
        if (C == 1) {
            mu = row_sum(red, 0, sum_t, 1u, nwarps, wwidth) * invN;
            const float d = mean_t - mu;
            const float m2 = row_sum(red, 1, fmaf(n_t * d, d, m2_t), 1u, nwarps, wwidth);
            rs = rsqrtf(m2 * invN + eps);
        } else if (Red::kWarpStates && nwarps * static_cast<int>(C) <= 32) {
            // At most 32 warps in the cluster: every warp merges its lanes'
            // states with butterflies and publishes its own (n, sum, M2);
            // one exchange through distributed shared memory then hands
            // lane l of every warp the state of warp l % nwarps of CTA
            // l / nwarps, and the warp merges the cluster's warp states by
            // the same rule. One barrier per row and no CTA-level pass.
            if constexpr (Red::kWarpStates) {
                const int lane = threadIdx.x & 31;
                const float n_w = group_sum(n_t, 32);
                const float s_w = group_sum(sum_t, 32);
                const float dw = mean_t - (n_w > 0.f ? s_w / n_w : 0.f);
                const float m2_w = group_sum(fmaf(n_t * dw, dw, m2_t), 32);
                if (lane == 0) red.warp_state[stage][threadIdx.x >> 5] = make_float4(n_w, s_w, m2_w, 0.f);
                cluster_barrier();
                float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
                if (lane < nwarps * static_cast<int>(C))
                    q = ld_peer_f32x4(peer_smem_addr(&red.warp_state[stage][lane % nwarps],
                                                     static_cast<uint32_t>(lane / nwarps)));
                mu = group_sum(q.y, 32) * invN;
                const float dq = (q.x > 0.f ? q.y / q.x : 0.f) - mu;
                const float m2 = group_sum(fmaf(q.x * dq, dq, q.z), 32);
                // every peer value consumed, the warp converged by the shuffles
                if constexpr (EARLY) cluster_arrive();  // the caller waits
                rs = rsqrtf(m2 * invN + eps);
            }
        } else {
            const float2 sn = cta_sum2(red, sum_t, n_t, nwarps, wwidth);  // this CTA's sum of x - K, count
            const float mean_c = sn.y > 0.f ? sn.x / sn.y : 0.f;
            const float dc = mean_t - mean_c;
            const float m2_c = row_sum(red, 1, fmaf(n_t * dc, dc, m2_t), 1u, nwarps, wwidth);
            float* st = red.cta_state[stage];
            if (threadIdx.x == 0) {
                st[0] = sn.y;
                st[1] = sn.x;
                st[2] = m2_c;
            }
            cluster_barrier();
            const int lane = threadIdx.x & 31;
            float nq = 0.f, sq = 0.f, mq = 0.f;
            if (lane < static_cast<int>(C)) {
                const uint32_t q = peer_smem_addr(st, static_cast<uint32_t>(lane));
                nq = ld_peer_f32(q);
                sq = ld_peer_f32(q + 4u);
                mq = ld_peer_f32(q + 8u);
            }
            mu = sum_first_lanes(sq, static_cast<int>(C)) * invN;
            const float dq = (nq > 0.f ? sq / nq : 0.f) - mu;
            const float m2 = sum_first_lanes(fmaf(nq * dq, dq, mq), static_cast<int>(C));
            // every peer value consumed, the warp converged by the shuffles
            if constexpr (EARLY) cluster_arrive();  // the caller waits
            rs = rsqrtf(m2 * invN + eps);
        }
    } else {
        mu = 0.f;
        rs = rsqrtf(row_sum<EARLY>(red, stage, ss_t, C, nwarps, wwidth) * invN + eps);
    }
}

// ================================================================== GROUP
// Lanes [k*G, (k+1)*G) of the CTA own row blockIdx*rows_per_cta + k. Lane l
// of a group holds accesses l, l+G, l+2G, ... (the G lanes of a group read G
// consecutive accesses per instruction). The statistics meet in xor
// butterflies over the group. ADD as for norm_fwd_cta.
template <class T, int VEC, int V, bool LN, bool ADD, bool Q8>
__global__ void __launch_bounds__(ADD ? kFusedMaxThreads : 1024) norm_fwd_group(const NormArgs a) {
    using S = Slice<T, VEC, V, LN>;
    const int G = a.group;
    const int tid = threadIdx.x;
    const int gl = tid & (G - 1);
    const int rows_per_cta = blockDim.x / G;
    const int nacc = (a.N + VEC - 1) / VEC;
    const int stride = G * VEC;
    const int nvalid = valid_runs(nacc, gl, G, V);
    const float n_t = static_cast<float>(nvalid * VEC);
    const float inv_n = nvalid > 0 ? 1.f / n_t : 0.f;
    const float invN = 1.f / static_cast<float>(a.N);
    const T* g = static_cast<const T*>(a.gamma) + gl * VEC;
    const T* b = static_cast<const T*>(a.beta) + gl * VEC;
    grid_release();
    grid_wait();
    const float inv = Q8 ? 1.f / *a.qscale : 0.f;

    for (int64_t rb = blockIdx.x; rb * rows_per_cta < a.M; rb += gridDim.x) {
        const int64_t row = rb * rows_per_cta + tid / G;
        const bool row_ok = row < a.M;
        const int nv = row_ok ? nvalid : 0;
        const T* xr = static_cast<const T*>(a.x) + row * a.ldx;
        const T* rr = ADD ? static_cast<const T*>(a.res) + row * a.N : nullptr;
        S s;
        const float K = (LN && row_ok) ? (ADD ? first_elem_add(xr, rr) : first_elem(xr)) : 0.f;
        s.set_shift(K);
        if constexpr (ADD)
            s.load_add(xr + gl * VEC, rr + gl * VEC, stride, nv);
        else
            s.load(xr + gl * VEC, stride, nv);
        float mu = 0.f, rs;
        if constexpr (LN) {
            float sum = 0.f, mean = 0.f, m2 = 0.f;
            s.template welford<!ADD>(nv, inv_n, sum, mean, m2);
            mu = group_sum(sum, G) * invN;
            const float d = mean - mu;
            const float M2 = group_sum(nv > 0 ? fmaf(n_t * d, d, m2) : 0.f, G);
            rs = rsqrtf(M2 * invN + a.eps);
            if (gl == 0 && row_ok) {
                if (a.mean) a.mean[row] = K + mu;
                if (a.rstd) a.rstd[row] = rs;
            }
        } else {
            rs = rsqrtf(group_sum(s.sumsq(nv), G) * invN + a.eps);
        }
        s.template out<Q8>(g, b, a.y, row * a.ldy + gl * VEC, stride, nv, mu, rs, inv);
        if constexpr (ADD) s.store_h(static_cast<T*>(a.h) + row * a.N + gl * VEC, stride, nv);
    }
}

// ================================================================== CTA
// A cluster of C CTAs (C = 1 without a cluster launch) owns one row per
// iteration. Round r of the row is the slice of accesses
// [(r*C + k)*V*T, (r*C + k + 1)*V*T) for CTA rank k, laid out warp-major.
// With one round the slice stays in registers from load to store. With
// several rounds each round is read for the statistics (its Welford state
// folded into the thread's state with the pairwise merge); the output pass
// then walks the rounds backwards, reusing the registers of the last round
// and re-reading the others. CL: launched with clusters (C > 1); without,
// every cluster step compiles away.
// ADD: fused residual add; the row is h = x + r (rounded to T). The rounds
// are then read in reverse, so that round 0, which holds the shift element
// every thread of the row reads first, is the one kept in registers; its h
// is stored in the output pass, after the row's barrier. The other rounds
// store h as soon as it is formed and the output pass re-reads h, not x and
// r. Every thread re-reads only its own accesses, so h (and y) may be the x
// or r buffer itself.
// Bulk L2 prefetch of the share of row `row` of x that CTA `rank` of a row's
// `C` CTAs reads: per round, `slots` 16-byte accesses at (round*C + rank) *
// slots from the start of the row's vector body (its first 16-byte aligned
// element), clipped to the row's whole vectors. No register is written and
// nothing waits for it.
template <class T, int VEC, bool SHIFT>
__device__ __forceinline__ void prefetch_row_share(const NormArgs& a, int64_t row, int rank, int C, int slots) {
    const T* xr = static_cast<const T*>(a.x) + row * a.ldx;
    int h0 = 0;
    if constexpr (SHIFT) {
        const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(xr)) & 15u;
        h0 = min(static_cast<int>(((16u - mis) & 15u) / sizeof(T)), a.N);
    }
    const int nb = (a.N - h0) / VEC;
    for (int r = 0; r < a.rounds; ++r) {
        const int f0 = (r * C + rank) * slots;
        const int n = min(slots, nb - f0);
        if (n > 0) prefetch_l2_bulk(xr + h0 + static_cast<int64_t>(f0) * VEC, static_cast<uint32_t>(n) * 16u);
    }
}

// FULL: one CTA per row in one round whose accesses exactly cover the row
// (N == threads * V * VEC; no cluster, no shift): every access of every
// thread is valid, so the accesses carry no bounds predicates. (The round
// count stays a runtime value: with both known, ptxas spilled the 16-bit
// LayerNorm variants at the 64-register cap.)
template <class T, int VEC, int V, bool LN, bool CL, bool ADD, bool Q8, bool SHIFT, bool FULL>
__global__ void __launch_bounds__(ADD ? kFusedMaxThreads : 1024) norm_fwd_cta(const NormArgs a) {
    static_assert(!FULL || (!CL && !SHIFT && VEC > 1), "FULL rows: one CTA, 16-byte vectors, no shift");
    using S = Slice<T, VEC, V, LN>;
    using SO = ScalarOps<T>;
    __shared__ std::conditional_t<CL, RowReduceSmemCl, RowReduceSmem> red;

    if constexpr (!ADD && VEC > 1) {
        // L2 prefetch of this CTA's share of the row a.group - 1 rows after
        // its first (a.group set at launch; 0: none): one CTA per row
        // prefetches a row that a CTA about to start will read, a cluster
        // its own row. It only moves data towards L2, so it runs before the
        // previous grid has finished (L2 is where that grid's writes land).
        if (threadIdx.x == 0 && a.group > 0) {
            const uint32_t cn = CL ? cluster_size() : 1u;
            const int64_t target = static_cast<int64_t>(blockIdx.x / cn) + (a.group - 1);
            if (target < a.M)
                prefetch_row_share<T, VEC, SHIFT>(a, target, CL ? static_cast<int>(cluster_rank()) : 0,
                                                  static_cast<int>(cn), V * static_cast<int>(blockDim.x));
        }
    }
    const int T_ = blockDim.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T_ >> 5;
    int wwidth = 1;  // power of two >= the number of warps
    while (wwidth < nwarps) wwidth <<= 1;
    const uint32_t C = CL ? cluster_size() : 1u;  // compile-time 1 without a cluster
    const int rank = CL ? static_cast<int>(cluster_rank()) : 0;
    const int64_t first_row = blockIdx.x / C;
    const int64_t row_step = gridDim.x / C;
    const int nacc = (a.N + VEC - 1) / VEC;
    const int rounds = a.rounds;
    const int stride = 32 * VEC;
    const int in_slice = warp * V * 32 + lane;  // this thread's first access within a slice
    const float invN = 1.f / static_cast<float>(a.N);
    // Fused add over a cluster, at most two accesses per thread and round
    // (what its planner picks): x and r evict first from L1 and the output
    // pass re-reads h without allocating in L1 (A/B on GB300, 2048x65536
    // fp32: + LayerNorm 357.1 -> 345.1 us, + RMSNorm 342.5 -> 338.1 us; one
    // CTA per row they lose up to 5 %, except 16-bit rows of two rounds).
    constexpr bool hint = ADD && CL && V <= 2;
    grid_release();
    grid_wait();
    const float inv = Q8 ? 1.f / *a.qscale : 0.f;

    for (int64_t row = first_row; row < a.M; row += row_step) {
        const T* xr = static_cast<const T*>(a.x) + row * a.ldx;
        const T* rr = ADD ? static_cast<const T*>(a.res) + row * a.N : nullptr;
        S s;
        const float K = LN ? (ADD ? first_elem_add(xr, rr) : first_elem(xr)) : 0.f;
        s.set_shift(K);
        T* hr = ADD ? static_cast<T*>(a.h) + row * a.N : nullptr;
        // SHIFT: the row's vectors start at its first 16-byte aligned element
        // h0; the h0 elements before them and the tail after the last whole
        // vector (together fewer than 2*VEC) are taken one per thread by the
        // first threads of CTA rank 0 (xi: the element, xraw its value).
        int h0 = 0, nb = nacc;
        bool sp = false;  // gamma/beta vectors not 16-byte aligned in this row
        int xi = -1;
        typename SO::Raw xraw = 0;
        if constexpr (SHIFT) {
            const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(xr)) & 15u;
            h0 = min(static_cast<int>(((16u - mis) & 15u) / sizeof(T)), a.N);
            nb = (a.N - h0) / VEC;
            sp = h0 != 0 || !a.vec_params;
            const int nextra = a.N - nb * VEC;
            if (rank == 0 && tid < nextra) {
                xi = tid < h0 ? tid : h0 + nb * VEC + (tid - h0);
                xraw = ADD ? SO::add_round(SO::load(xr + xi), SO::load(rr + xi)) : SO::load(xr + xi);
            }
        }
        const T* xb = xr + h0;  // the row's vector body
        const T* rb = ADD ? rr + h0 : nullptr;
        T* hb = ADD ? hr + h0 : nullptr;
        float n_t = 0.f, sum_t = 0.f, mean_t = 0.f, m2_t = 0.f, ss_t = 0.f;
        int nv = 0;
        for (int i = 0; i < rounds; ++i) {
            const int r = ADD ? rounds - 1 - i : i;
            const int f = (r * static_cast<int>(C) + rank) * V * T_ + in_slice;
            nv = FULL ? V : valid_runs(nb, f, 32, V);
            if constexpr (ADD) {
                s.template load_add<hint>(xb + f * VEC, rb + f * VEC, stride, nv);
                if (r != 0) s.store_h(hb + f * VEC, stride, nv);
            } else {
                s.load(xb + f * VEC, stride, nv);
            }
            if constexpr (LN) {
                const float n = static_cast<float>(nv * VEC);
                float sum = 0.f, mean = 0.f, m2 = 0.f;
                s.template welford<!ADD && !CL>(nv, nv > 0 ? 1.f / n : 0.f, sum, mean, m2);
                if (i == 0) {
                    n_t = n, sum_t = sum, mean_t = mean, m2_t = m2;
                } else if (n > 0.f) {  // pairwise merge ([Ch7] §7.4.1)
                    const float nn = n_t + n;
                    const float wb = n / nn;
                    const float d = mean - mean_t;
                    m2_t = m2_t + m2 + d * d * n_t * wb;
                    mean_t = fmaf(d, wb, mean_t);
                    sum_t += sum;
                    n_t = nn;
                }
            } else {
                ss_t += s.sumsq(nv);
            }
        }
        if constexpr (SHIFT) {
            if (xi >= 0) {  // fold the extra element in: the one-element update ([Ch7] §7.4)
                const float xe = SO::e(xraw);
                if constexpr (LN) {
                    const float d0 = xe - K;
                    const float n1 = n_t + 1.f;
                    const float d = d0 - mean_t;
                    mean_t += d / n1;
                    m2_t = fmaf(d, d0 - mean_t, m2_t);
                    sum_t += d0;
                    n_t = n1;
                } else {
                    ss_t = fmaf(xe, xe, ss_t);
                }
            }
        }
        float mu, rs;
        row_stats<LN, CL>(red, n_t, sum_t, mean_t, m2_t, ss_t, invN, a.eps, C, nwarps, wwidth, 0, mu, rs);
        if (LN && rank == 0 && tid == 0) {
            if (a.mean) a.mean[row] = K + mu;
            if (a.rstd) a.rstd[row] = rs;
        }
        const T* gb = static_cast<const T*>(a.gamma) + h0;
        const T* bb = static_cast<const T*>(a.beta) + h0;
        const int64_t yb = row * a.ldy + h0;
        if constexpr (SHIFT) {
            if (xi >= 0) {  // the extra element's output (and h), after the row's barrier
                const T* g1 = static_cast<const T*>(a.gamma) + xi;
                const float nmr = -mu * rs;
                if constexpr (Q8) {
                    float o;
                    if constexpr (LN)
                        SO::ln_vals(xraw, K, rs, nmr, SO::load_param(g1), SO::load_param(static_cast<const T*>(a.beta) + xi),
                                    &o);
                    else
                        SO::rms_vals(xraw, rs, SO::load_param(g1), &o);
                    store_e4m3<1>(static_cast<uint8_t*>(a.y) + row * a.ldy + xi, &o, inv);
                } else {
                    T* y1 = static_cast<T*>(a.y) + row * a.ldy + xi;
                    if constexpr (LN)
                        SO::store(y1, SO::ln_out(xraw, K, rs, nmr, SO::load_param(g1),
                                                 SO::load_param(static_cast<const T*>(a.beta) + xi)));
                    else
                        SO::store(y1, SO::rms_out(xraw, rs, SO::load_param(g1)));
                }
                if constexpr (ADD) SO::store(hr + xi, xraw);
            }
        }
        if constexpr (ADD) {
            for (int r = 0; r < rounds; ++r) {
                const int f = (r * static_cast<int>(C) + rank) * V * T_ + in_slice;
                if (r != 0) {
                    nv = FULL ? V : valid_runs(nb, f, 32, V);
                    s.template load<hint>(hb + f * VEC, stride, nv);  // only this thread wrote h there
                }
                s.template out<Q8>(gb + f * VEC, bb + f * VEC, a.y, yb + f * VEC, stride, nv, mu, rs, inv, sp);
                if (r == 0) s.store_h(hb + f * VEC, stride, nv);
            }
        } else {
            for (int r = rounds - 1; r >= 0; --r) {
                const int f = (r * static_cast<int>(C) + rank) * V * T_ + in_slice;
                if (r != rounds - 1) {
                    nv = FULL ? V : valid_runs(nb, f, 32, V);
                    s.load(xb + f * VEC, stride, nv);
                }
                s.template out<Q8>(gb + f * VEC, bb + f * VEC, a.y, yb + f * VEC, stride, nv, mu, rs, inv, sp);
            }
        }
        // RMSNorm reduces once per row, always in stage 0, and a LayerNorm
        // cluster publishes its CTA state once per row, in stage 0: before
        // this CTA (cluster) writes that slot again for its next row, every
        // thread of it (and of its peers) must have read this row's values.
        // (One CTA's LayerNorm sums use two stages and order that by
        // themselves.) One-row-per-CTA launches never get here. In a
        // cluster every thread arrived right after reading its peers'
        // values (row_stats, EARLY), so the wait here is for the peers'
        // reads only, not for their output passes.
        if constexpr (!LN || CL) {
            if (row + row_step < a.M) {
                if (C > 1)
                    cluster_wait();
                else
                    __syncthreads();
            }
        }
    }
    // No CTA may exit while a peer can still read its shared memory: wait
    // on the arrive of the last row's exchange (CTAs of a cluster share
    // their rows, so a cluster without rows made no exchange at all).
    if (C > 1 && first_row < a.M) cluster_wait();
}

// ================================================================== RING
// fp32 pair arithmetic: the packed sm_100-family instructions for 16-bit
// rows, scalar instructions for fp32 rows (as in the register kernels).
template <bool PACKED>
struct PairMath;
template <>
struct PairMath<true> {
    static __device__ __forceinline__ float2 add(float2 a, float2 b) { return __fadd2_rn(a, b); }
    static __device__ __forceinline__ float2 mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
    static __device__ __forceinline__ float2 fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
};
template <>
struct PairMath<false> {
    static __device__ __forceinline__ float2 add(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
    static __device__ __forceinline__ float2 mul(float2 a, float2 b) { return make_float2(a.x * b.x, a.y * b.y); }
    static __device__ __forceinline__ float2 fma(float2 a, float2 b, float2 c) {
        return make_float2(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y));
    }
};

// Element pair i of a 16-byte access, widened exactly to fp32, and the
// reverse (nearest-even rounding to T).
template <class T>
struct PairCodec {
    using P = typename std::conditional<std::is_same<T, __half>::value, F16Pair, Bf16Pair>::type;
    static __device__ __forceinline__ float2 get(const uint4& r, int i) {
        if constexpr (sizeof(T) == 4)
            return i == 0 ? make_float2(__uint_as_float(r.x), __uint_as_float(r.y))
                          : make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
        else
            return P::widen(i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w);
    }
    static __device__ __forceinline__ uint4 put(const float2* v) {
        if constexpr (sizeof(T) == 4)
            return make_uint4(__float_as_uint(v[0].x), __float_as_uint(v[0].y), __float_as_uint(v[1].x),
                              __float_as_uint(v[1].y));
        else
            return make_uint4(P::pack(v[0].x, v[0].y), P::pack(v[1].x, v[1].y), P::pack(v[2].x, v[2].y),
                              P::pack(v[3].x, v[3].y));
    }
    // The first element of a 16-byte access.
    static __device__ __forceinline__ float first(const uint4& r) { return get(r, 0).x; }
};

// A thread's V accesses of one row, widened once to fp32 pairs and kept in
// registers: x - K for LayerNorm, x for RMSNorm. The first `nvalid` lie
// inside the row. Every value is the one the register kernels form at each
// use (x - K is rounded the same way), so the two statistics passes and the
// output step read them without widening again.
template <class T, int V, bool LN>
struct WideSlice {
    static constexpr int VEC = ElemVec<T>::value;
    static constexpr int NP = VEC / 2;  // fp32 pairs per access
    using PM = PairMath<sizeof(T) == 2>;
    using PC = PairCodec<T>;
    float2 d[V][NP];

    __device__ __forceinline__ void set(int j, const uint4& r, float2 nk) {
#pragma unroll
        for (int i = 0; i < NP; ++i) d[j][i] = LN ? PM::add(PC::get(r, i), nk) : PC::get(r, i);
    }
    // Welford state of the valid elements ([Ch7] §7.4): the sum and mean of
    // x - K, then M2 about that mean, two passes over the registers.
    __device__ __forceinline__ void welford(int nvalid, float inv_n, float& sum, float& mean, float& m2) const {
        float2 s0 = make_float2(0.f, 0.f), s1 = s0;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    if (i & 1)
                        s1 = PM::add(s1, d[j][i]);
                    else
                        s0 = PM::add(s0, d[j][i]);
                }
            }
        const float2 s = PM::add(s0, s1);
        sum = s.x + s.y;
        mean = sum * inv_n;
        const float2 nm = f2_splat(-mean);
        float2 q0 = make_float2(0.f, 0.f), q1 = q0;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    const float2 e = PM::add(d[j][i], nm);
                    if (i & 1)
                        q1 = PM::fma(e, e, q1);
                    else
                        q0 = PM::fma(e, e, q0);
                }
            }
        const float2 q = PM::add(q0, q1);
        m2 = q.x + q.y;
    }
    // Sum of squares of the valid elements (RMSNorm, [Ch7] §7.5.1).
    __device__ __forceinline__ float sumsq(int nvalid) const {
        float2 q0 = make_float2(0.f, 0.f), q1 = q0;
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    if (i & 1)
                        q1 = PM::fma(d[j][i], d[j][i], q1);
                    else
                        q0 = PM::fma(d[j][i], d[j][i], q0);
                }
            }
        const float2 q = PM::add(q0, q1);
        return q.x + q.y;
    }
    // y = ((x - K) * rstd - mu * rstd) * gamma + beta (LayerNorm) or
    // (x * w) * rstd (RMSNorm), rounded to T and stored; `g`, `b` and `y`
    // point at this thread's first access, `stride` elements apart.
    __device__ __forceinline__ void emit(const T* g, const T* b, T* y, int stride, int nvalid, float mu,
                                         float rs) const {
        const float2 rs2 = f2_splat(rs), nm2 = f2_splat(-mu * rs);
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) {
                const uint4 gr = __ldg(reinterpret_cast<const uint4*>(g + j * stride));
                uint4 br = make_uint4(0u, 0u, 0u, 0u);
                if constexpr (LN) br = __ldg(reinterpret_cast<const uint4*>(b + j * stride));
                float2 o[NP];
#pragma unroll
                for (int i = 0; i < NP; ++i)
                    o[i] = LN ? PM::fma(PM::fma(d[j][i], rs2, nm2), PC::get(gr, i), PC::get(br, i))
                              : PM::mul(PM::mul(d[j][i], PC::get(gr, i)), rs2);
                *reinterpret_cast<uint4*>(y + j * stride) = PC::put(o);
            }
    }
};

// The CTA mapping (one CTA or cluster per row, one round) on a persistent
// grid. A CTA's share of a row is one contiguous run of V*T accesses (the
// warp-major layout), so thread 0 moves it into shared memory with a
// single bulk copy, counted on the stage's mbarrier; a ring of `stages`
// such stages keeps this CTA's next rows in flight while it reduces and
// stores the current one. Each thread widens its accesses from its stage
// once (WideSlice) and works from registers. A stage is refilled, with the
// row `stages` steps ahead, right after the current row's statistics: the
// barriers of that reduction come after every thread's reads of the stage.
// LayerNorm's shift K (the row's first element) arrives with each stage in
// a 16-byte slot of its own, so every CTA of a cluster has it. Needs
// 16-byte aligned rows of whole vectors.
template <class T, int V, bool LN, bool CL>
__global__ void __launch_bounds__(kRingMaxThreads) norm_fwd_ring(const NormArgs a) {
    constexpr int VEC = ElemVec<T>::value;
    using S = WideSlice<T, V, LN>;
    // [stages][V*T] 16-byte slots | [stages] first 16 bytes of the row | [stages] mbarriers
    extern __shared__ __align__(128) uint4 ring[];
    __shared__ std::conditional_t<CL, RowReduceSmemCl, RowReduceSmem> red;

    const int stages = a.stages;
    const int T_ = blockDim.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T_ >> 5;
    int wwidth = 1;
    while (wwidth < nwarps) wwidth <<= 1;
    const uint32_t C = CL ? cluster_size() : 1u;  // compile-time 1 without a cluster
    const int rank = CL ? static_cast<int>(cluster_rank()) : 0;
    const int64_t first_row = blockIdx.x / C;
    const int64_t row_step = gridDim.x / C;
    const int nacc = a.N / VEC;
    const int stride = 32 * VEC;
    const int stage_slots = V * T_;
    const int cbase = rank * stage_slots;  // this CTA's first access of every row
    const int cslots = max(0, min(stage_slots, nacc - cbase));
    const uint32_t cbytes = static_cast<uint32_t>(cslots) * 16u;
    const uint32_t tx = cbytes + (LN ? 16u : 0u);
    const int in_slice = warp * V * 32 + lane;
    const int nvalid = valid_runs(cslots, in_slice, 32, V);
    const float n_t = static_cast<float>(nvalid * VEC);
    const float inv_n = nvalid > 0 ? 1.f / n_t : 0.f;
    const float invN = 1.f / static_cast<float>(a.N);
    uint4* kslot = ring + stages * stage_slots;
    uint64_t* full = reinterpret_cast<uint64_t*>(kslot + stages);
    const T* x = static_cast<const T*>(a.x);
    const int64_t col = static_cast<int64_t>(cbase + in_slice) * VEC;  // this thread's first element
    const T* g = static_cast<const T*>(a.gamma) + col;
    const T* b = static_cast<const T*>(a.beta) + col;

    // Set by any thread whose wait for a stage ran out. Every thread reads
    // it before its next wait, and thread 0 before its next copy, each after
    // the barrier of the row reduction that follows the wait: from the row
    // after a timeout on, the whole CTA neither waits nor copies.
    __shared__ int s_late;
    if (tid == 0) {
        for (int k = 0; k < stages; ++k) mbar_init(&full[k], 1);
        mbar_init_fence();
        s_late = 0;
    }
    __syncthreads();
    grid_release();
    grid_wait();
    const uint64_t limit = a.wait->limit_ns;

    // Thread 0: fill stage `st` with this CTA's share of `row`.
    auto issue = [&](int64_t row, int st) {
        const T* xr = x + row * a.ldx;
        mbar_arrive_expect(&full[st], tx);
        if (cbytes) bulk_load(ring + st * stage_slots, xr + cbase * VEC, cbytes, &full[st]);
        if (LN) bulk_load(kslot + st, xr, 16u, &full[st]);
    };
    int64_t issued = 0;  // thread 0: rows of this CTA whose copies it issued
    if (tid == 0)
        for (int k = 0; k < stages; ++k)
            if (first_row + k * row_step < a.M) {
                issue(first_row + k * row_step, k);
                ++issued;
            }

    volatile int& late = s_late;
    int st = 0;
    uint32_t parity = 0;
    int64_t k = 0;        // rows of this CTA done so far
    int64_t seen = 0;     // thread 0: leading rows whose copies it saw complete
    bool waiting = true;  // this thread still waits for its stages
    for (int64_t row = first_row; row < a.M; row += row_step, ++k) {
        // After a wait has run out the CTA neither waits nor copies any more
        // (its outputs are void by then), so the kernel still ends in
        // bounded time.
        if (waiting) {
            if (late)
                waiting = false;
            else if (!mbar_wait(&full[st], parity, limit))
                late = 1, waiting = false;
            else
                seen = k + 1;
        }
        float K = 0.f;
        if constexpr (LN) K = PairCodec<T>::first(kslot[st]);
        S s;
        const uint4* src = ring + st * stage_slots + in_slice;
        const float2 nk = f2_splat(-K);
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < nvalid) s.set(j, src[j * 32], nk);
        float sum = 0.f, mean = 0.f, m2 = 0.f, ss = 0.f;
        if constexpr (LN)
            s.welford(nvalid, inv_n, sum, mean, m2);
        else
            ss = s.sumsq(nvalid);
        float mu, rs;
        row_stats<LN>(red, n_t, sum, mean, m2, ss, invN, a.eps, C, nwarps, wwidth, static_cast<int>(k & 1), mu, rs);
        if (LN && rank == 0 && tid == 0) {
            if (a.mean) a.mean[row] = K + mu;
            if (a.rstd) a.rstd[row] = rs;
        }
        if (tid == 0 && !late) {
            const int64_t next = row + stages * row_step;
            if (next < a.M) {
                fence_proxy_async();
                issue(next, st);
                ++issued;
            }
        }
        s.emit(g, b, static_cast<T*>(a.y) + row * a.ldy + col, stride, nvalid, mu, rs);
        if (++st == stages) st = 0, parity ^= 1u;
    }
    if (tid == 0 && late) {
        // Copies that may still be in flight (the rows issued after the last
        // one thread 0 saw complete; a stage is refilled only after its
        // previous row completed, so each has one outstanding phase) get one
        // more wait each, with the full limit, so that none lands after this
        // CTA has gone; then tell the host.
        for (int64_t kk = seen; kk < issued; ++kk)
            mbar_wait(&full[kk % stages], static_cast<uint32_t>((kk / stages) & 1), kDefaultWaitLimitNs);
        atomicAdd(&a.wait->timeouts, 1u);
    }
    // No CTA may exit while a peer can still read its shared memory.
    if (C > 1) cluster_barrier();
}

// ================================================================== launch
template <class T, bool LN>
using KernelFn = void (*)(const NormArgs);

// SHIFT variants exist for the 16-byte vector width only (element rows
// need no alignment).
template <class T, bool LN, bool ADD, bool Q8, int VEC, int V>
KernelFn<T, LN> pick_cta(bool cl, bool shift, bool full) {
    if constexpr (VEC > 1) {
        if (shift)
            return cl ? norm_fwd_cta<T, VEC, V, LN, true, ADD, Q8, true, false>
                      : norm_fwd_cta<T, VEC, V, LN, false, ADD, Q8, true, false>;
        if constexpr (Q8) {
            if (full && !cl) return norm_fwd_cta<T, VEC, V, LN, false, ADD, Q8, false, true>;
        }
    }
    return cl ? norm_fwd_cta<T, VEC, V, LN, true, ADD, Q8, false, false>
              : norm_fwd_cta<T, VEC, V, LN, false, ADD, Q8, false, false>;
}

template <class T, bool LN, bool ADD, bool Q8, int VEC>
KernelFn<T, LN> pick_kernel(int mapping, int per_thread, bool cl, bool shift, bool full) {
    const bool group = mapping == NORM_MAP_GROUP;
    switch (per_thread) {
        case 1: return group ? norm_fwd_group<T, VEC, 1, LN, ADD, Q8> : pick_cta<T, LN, ADD, Q8, VEC, 1>(cl, shift, full);
        case 2: return group ? norm_fwd_group<T, VEC, 2, LN, ADD, Q8> : pick_cta<T, LN, ADD, Q8, VEC, 2>(cl, shift, full);
        case 4: return group ? norm_fwd_group<T, VEC, 4, LN, ADD, Q8> : pick_cta<T, LN, ADD, Q8, VEC, 4>(cl, shift, full);
        case 8: return group ? norm_fwd_group<T, VEC, 8, LN, ADD, Q8> : pick_cta<T, LN, ADD, Q8, VEC, 8>(cl, shift, full);
        default: return nullptr;
    }
}

template <class T, bool LN, int V>
KernelFn<T, LN> pick_ring_v(bool cl) {
    return cl ? norm_fwd_ring<T, V, LN, true> : norm_fwd_ring<T, V, LN, false>;
}

template <class T, bool LN>
KernelFn<T, LN> pick_ring(int per_thread, bool cl) {
    switch (per_thread) {
        case 1: return pick_ring_v<T, LN, 1>(cl);
        case 2: return pick_ring_v<T, LN, 2>(cl);
        case 4: return pick_ring_v<T, LN, 4>(cl);
        case 8: return pick_ring_v<T, LN, 8>(cl);
        default: return nullptr;
    }
}

// Opt a ring kernel in to the device's largest dynamic shared memory
// per block (once per kernel and device; the call is not a stream operation).
template <class T, int V, bool LN, bool CL>
cudaError_t opt_in_smem(int dev) {
    static std::atomic<unsigned long long> done{0};
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    if (bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, norm_fwd_ring<T, V, LN, CL>);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(norm_fwd_ring<T, V, LN, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(fa.sharedSizeBytes));
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

template <class T, bool LN, int V>
cudaError_t allow_smem_v(bool cl, int dev) {
    return cl ? opt_in_smem<T, V, LN, true>(dev) : opt_in_smem<T, V, LN, false>(dev);
}

template <class T, bool LN>
cudaError_t allow_smem(int per_thread, bool cl, int dev) {
    switch (per_thread) {
        case 1: return allow_smem_v<T, LN, 1>(cl, dev);
        case 2: return allow_smem_v<T, LN, 2>(cl, dev);
        case 4: return allow_smem_v<T, LN, 4>(cl, dev);
        case 8: return allow_smem_v<T, LN, 8>(cl, dev);
        default: return cudaErrorInvalidValue;
    }
}

// CTAs of kernel `k` with `threads` threads (no dynamic shared memory) that
// fit on device `dev` at once; queried once per kernel, size and device.
inline cudaError_t resident_ctas(const void* k, int threads, int dev, int num_sms, int64_t* out) {
    struct Key {
        const void* fn;
        int threads, dev;
        bool operator<(const Key& o) const { return std::tie(fn, threads, dev) < std::tie(o.fn, o.threads, o.dev); }
    };
    static std::mutex mu;
    static std::map<Key, int64_t> cache;
    const Key key{k, threads, dev};
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, 0);
    if (e != cudaSuccess) return e;
    cache[key] = int64_t(n) * num_sms;
    *out = cache[key];
    return cudaSuccess;
}

// Rows at least this long (bytes of x) get the next-row L2 prefetch.
constexpr int64_t kPrefetchMinRowBytes = 8192;

// ADD: the fused residual add; Q8: FP8 E4M3 output (register kernels only;
// no ring).
template <class T, bool LN, bool ADD, bool Q8 = false>
cudaError_t launch_norm(const norm_plan& p, const NormArgs& a, cudaStream_t stream, int num_sms, int dev) {
    KernelFn<T, LN> k;
    size_t smem = 0;
    const bool cl = p.mapping == NORM_MAP_CTA && p.cluster > 1;
    if (p.stages > 0) {
        if constexpr (ADD || Q8) {
            return cudaErrorInvalidValue;
        } else {
            k = pick_ring<T, LN>(p.per_thread, cl);
            if (k == nullptr) return cudaErrorInvalidValue;
            smem = ring_smem_bytes(p.stages, p.per_thread, p.threads);
            const cudaError_t e = allow_smem<T, LN>(p.per_thread, cl, dev);
            if (e != cudaSuccess) return e;
        }
    } else {
        // Rows exactly covered by one round of one CTA's accesses, FP8
        // output only (A/B on GB300: FP8 LayerNorm bf16 4096x8192 21.67 ->
        // 20.98 us; the row-dtype outputs measured slower without the
        // predicates, LayerNorm bf16 21.78 -> 22.73 us).
        const bool full = Q8 && p.mapping == NORM_MAP_CTA && p.cluster == 1 && p.rounds == 1 && a.shift == 0 &&
                          p.vec_elems > 1 && int64_t(a.N) == int64_t(p.threads) * p.per_thread * p.vec_elems;
        k = p.vec_elems == 1 ? pick_kernel<T, LN, ADD, Q8, 1>(p.mapping, p.per_thread, cl, false, false)
                             : pick_kernel<T, LN, ADD, Q8, ElemVec<T>::value>(p.mapping, p.per_thread, cl,
                                                                               a.shift != 0, full);
        if (k == nullptr) return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(p.threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.mapping == NORM_MAP_CTA && p.cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(p.cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    NormArgs args = a;
    if (!ADD && p.mapping == NORM_MAP_CTA && p.stages == 0 && p.vec_elems > 1) {
        // L2 prefetch (args.group = rows ahead + 1). One CTA per row, rows of
        // at least kPrefetchMinRowBytes: the row 3/8 of the resident CTAs
        // ahead for fp32 rows, 1/4 for 16-bit rows, just past the rows in
        // flight (measured on GB300: 1/4 to 1/2 ahead gain 2-14 %, a whole
        // resident set ahead loses; 1/4 instead of 3/8 on 16-bit rows:
        // LayerNorm bf16 4096x8192 21.82 -> 21.39 us, fp16 21.86 -> 21.61 us,
        // 16384x8192 and RMSNorm bf16 8192x8192 unchanged; on fp32 rows 3/8
        // stays ahead, LayerNorm fp32 8192x5000 46.71 against 46.89 us at
        // 1/4). A cluster per
        // row: its own row (a row ahead loses at any distance; its own row
        // gains 2.6 % on 65536-wide rows). A launch whose rows all fit in one
        // wave of resident CTAs: each CTA its own row, so that the fetch
        // overlaps the previous grid's tail. The fused add measured slower
        // with it and has none.
        if (p.cluster > 1) {
            args.group = 1;
        } else {
            int64_t resident = 0;
            const cudaError_t e = resident_ctas(reinterpret_cast<const void*>(k), p.threads, dev, num_sms, &resident);
            if (e != cudaSuccess) return e;
            if (a.M <= resident && p.grid >= a.M)
                args.group = 1;
            else if (int64_t(a.N) * int64_t(sizeof(T)) >= kPrefetchMinRowBytes)
                args.group = static_cast<int32_t>(std::min<int64_t>(resident * (sizeof(T) == 2 ? 2 : 3) / 8, a.M) + 1);
        }
    }
    if (p.stages > 0) {
        args.wait = wait_state(dev);
        if (args.wait == nullptr) return cudaErrorInvalidSymbol;
    }
    if (p.stages > 0 && p.grid == 0) {
        // Persistent grid: as many CTAs (whole clusters) as can be resident at
        // once, so that no row waits for a CTA that never finishes early.
        int64_t clusters;
        if (p.cluster > 1) {
            cfg.gridDim = dim3(static_cast<unsigned>(p.cluster), 1, 1);
            int n = 0;
            const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
            if (e != cudaSuccess) return e;
            clusters = n;
        } else {
            int per_sm = 0;
            const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, p.threads, smem);
            if (e != cudaSuccess) return e;
            clusters = int64_t(per_sm) * num_sms;
        }
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(a.M, clusters) * p.cluster), 1, 1);
    }
    return cudaLaunchKernelEx(&cfg, k, args);
}

}  // namespace libnorm
