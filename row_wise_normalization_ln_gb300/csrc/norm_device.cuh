// Device building blocks of the row-wise LayerNorm / RMSNorm forward kernels:
// warp xor-shuffle butterflies ([Ch7] §7.4.2), cluster (distributed shared
// memory) primitives, and per-thread asynchronous copies into shared memory.
//
// Source (page title, section): [Ch7] "第 7 章 LayerNorm 与 RMSNorm",
// §7.4.2 warp xor-shuffle reduction, §7.6 two-level block reduction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace libnorm {

constexpr unsigned kFullMask = 0xffffffffu;

// ----------------------------------------------------------------- butterflies
// Sum over aligned groups of `width` lanes (a power of two <= 32; every lane
// of the warp must call it). fp32 addition is commutative, so every lane of a
// group ends with the same bits.
__device__ __forceinline__ float group_sum(float v, int width) {
    for (int off = width >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(kFullMask, v, off);
    return v;
}

// Sum over lanes [0, width) (width a power of two), handed to every lane of
// the warp: a butterfly of log2(width) levels, then a broadcast from lane 0.
__device__ __forceinline__ float sum_first_lanes(float v, int width) {
    v = group_sum(v, width);
    return width < 32 ? __shfl_sync(kFullMask, v, 0) : v;
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

// The two halves of cluster_barrier, for a barrier whose arrival can come
// early: a thread arrives once it has finished the accesses its peers must
// see completed (its reads of their shared memory), does other work, and
// waits later, right before what those accesses must precede (a peer
// rewriting or releasing that memory). A thread's arrives and waits
// alternate; every CTA of the cluster makes the same sequence of them.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
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

__device__ __forceinline__ float4 ld_peer_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// ----------------------------------------------------------- dependent launch
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may be scheduled before the previous kernel
// in its stream has finished. `grid_wait` blocks until that previous grid has
// completed and its memory is visible (a no-op without such a dependency), so
// every kernel calls it before its first global memory access;
// `grid_release` lets the next such launch be scheduled once every CTA of
// this grid has issued it. Kernels launched without the attribute (any
// other library's) still wait for this grid to complete.
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_release() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ----------------------------------------------------------------- L2 prefetch
// Hints that move data towards L2 without writing any register, so nothing
// (no barrier, no scoreboard) waits for them: a bulk range through the copy
// engine (16-byte aligned address, size a multiple of 16), or one line.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ----------------------------------------------------------------- bulk copies
// One thread moves a contiguous global range into shared memory with a 1-D
// bulk copy (the Tensor Memory Accelerator's untiled form: both addresses
// 16-byte aligned, the size a multiple of 16). The copy counts its bytes
// against an mbarrier in the destination CTA: that thread first arrives on
// the barrier announcing the bytes to expect, and the barrier's phase
// completes once they have all landed. Readers wait for the phase, so every
// byte they read was written by the copy.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t arrivals) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(arrivals) : "memory");
}

// Makes initialised barriers visible to the copy engine (before any copy
// names them).
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Arrive once (release at CTA scope: this thread's earlier writes are
// visible to every thread that then sees the phase complete).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Asynchronous store of a float2 into a cluster peer's shared memory
// (`addr`, from mapa), counted as 8 bytes against the peer's mbarrier
// (`bar`, from mapa): the peer sees the value once that barrier's phase
// completes. Weakly ordered: no fence with this thread's other accesses.
__device__ __forceinline__ void st_async_peer_f32x2(uint32_t addr, float2 v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
                 "f"(v.x), "f"(v.y), "r"(bar)
                 : "memory");
}

// Arrive once, announcing `bytes` more bytes for the current phase.
__device__ __forceinline__ void mbar_arrive_expect(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// The same test without suspending: true if the phase has completed now.
__device__ __forceinline__ bool mbar_test_now(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the phase of parity `parity` of `bar` has completed; false if
// it has not within `limit_ns` nanoseconds of %globaltimer (the copies it
// waits for take microseconds). A limit of 0 tests once, without waiting.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_test_now(bar, parity)) return true;
    if (limit_ns == 0) return false;
    const uint64_t t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_test(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Copy `bytes` from global `src` to this CTA's shared `dst`, completing on
// `bar` (this CTA's).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Orders this thread's view of shared memory (including reads that a
// preceding barrier made complete for the whole CTA) before its next bulk
// copy into shared memory.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

}  // namespace libnorm
