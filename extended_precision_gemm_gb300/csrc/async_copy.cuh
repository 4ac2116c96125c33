// async_copy.cuh -- bulk asynchronous copies (TMA engine) into shared memory
// with mbarrier completion, and bounded waits on those barriers.
#pragma once

#include <cstdint>

namespace ddg {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (the copy engine).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of the barrier to complete, for at most `budget` ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long budget) {
    for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > budget) return false;
    }
}

// Plain arrive on a barrier of this CTA.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile(
        "{\n"
        " .reg .b64 st;\n"
        " mbarrier.arrive.shared::cta.b64 st, [%0];\n"
        "}\n" ::"r"(bar)
        : "memory");
}

// Arrive on the barrier at shared-memory offset `bar` of CTA `rank` of this
// cluster.  (The arrivals of the slice GEMM announce data the tensor core
// reads or tensor memory it may overwrite; no generic-proxy data is published
// through them, so the default semantics suffice and no cluster-scope fence
// is paid per arrival.)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
    asm volatile(
        "{\n"
        " .reg .b32 ra;\n"
        " mapa.shared::cluster.u32 ra, %0, %1;\n"
        " mbarrier.arrive.shared::cluster.b64 _, [ra];\n"
        "}\n" ::"r"(bar),
        "r"(rank)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Arrive on the barrier, announcing `bytes` of copies that will complete it.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n"
        " .reg .b64 st;\n"
        " mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n"
        "}\n" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Address of the shared-memory offset `local` of CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Tensor copy of the 2-D box at (x, y) of `tmap` into this CTA's shared
// memory; with cta_group::2 the completion (its bytes) may be signalled on a
// barrier of either CTA of the pair (`bar`: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

}  // namespace ddg
