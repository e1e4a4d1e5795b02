// Asynchronous-copy building blocks (sm_90+ PTX, used on sm_103a): mbarriers,
// 1-D bulk copies global -> shared (the TMA engine, cp.async.bulk) and a
// wait that is bounded by the global nanosecond timer.
//
// Each translation unit that includes this header gets its own device status
// word (internal linkage): bit 0 is set when a bounded wait runs out.  The
// unit exports a host function that reads it, and the C ABI ORs them.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rs {

namespace {
__device__ unsigned int g_unit_status;
}

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s per mbarrier wait
constexpr unsigned int kStatusWaitTimeout = 1u;

__device__ __forceinline__ void flag_timeout() { atomicOr(&g_unit_status, kStatusWaitTimeout); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the async proxy and the cluster.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory
// before its later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Raises the phase's expected transaction bytes without arriving (the phase
// cannot complete before the pending arrival, so copies may be announced one
// at a time).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from global to this CTA's shared
// memory; both addresses 16-byte aligned.  Completion (complete_tx) is
// signalled on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Cluster-scope variant: the phase's completion also makes the data that
// other CTAs of the cluster delivered with st.async visible to this thread.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Asynchronous 8-byte store into another CTA's shared memory (cluster
// address), counted as 8 transaction bytes on that CTA's mbarrier.
__device__ __forceinline__ void st_async_pair(uint32_t remote_addr, float a, float b, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(remote_addr),
        "f"(a), "f"(b), "r"(remote_bar)
        : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity to complete; false if
// that takes longer than limit_ns (default kWaitLimitNs).
static __device__ __noinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                      uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

static __device__ __noinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                              uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Host side: read (and optionally clear) this unit's status word.
static inline cudaError_t read_unit_status(unsigned int* flags, bool clear) {
    unsigned int v = 0;
    cudaError_t err = cudaMemcpyFromSymbol(&v, g_unit_status, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    *flags |= v;
    if (!clear) return cudaSuccess;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_unit_status, &zero, sizeof(unsigned int));
}

}  // namespace rs
