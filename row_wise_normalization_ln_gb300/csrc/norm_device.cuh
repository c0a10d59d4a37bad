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

// ----------------------------------------------------------------- cp.async
// Per-thread asynchronous global -> shared copies. A thread waits for its own
// copies with cp.async.wait_group, a hardware wait (no polling loop), and
// then reads what it copied; no other thread reads those bytes.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most `pending` (0..3) of this thread's newest copy groups
// are still in flight.
__device__ __forceinline__ void cp_async_wait(int pending) {
    switch (pending) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    }
}

}  // namespace libnorm
