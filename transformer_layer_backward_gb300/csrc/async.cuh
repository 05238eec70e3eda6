// Asynchronous-copy primitives of sm_100-class GPUs used by the streaming kernels:
// shared-memory mbarriers, bulk (TMA) copies global -> shared, proxy fences, and
// bounded waits.  Every wait has an iteration/clock limit: on timeout it records
// TLB_ETIMEOUT-class status in the workspace status block and returns false, so a
// kernel can wind down instead of hanging.
#pragma once

#include "common.cuh"

namespace tlb {

// ~1 s at 2 GHz: far beyond any legitimate wait of these kernels.
constexpr long long kWaitLimitCycles = 2000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Arrive on the barrier and announce `bytes` of transaction to come.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) from global to
// this CTA's shared memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_1d(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Record a device-side timeout (first one wins) in the workspace status block.
__device__ __forceinline__ void report_timeout(uint32_t *status, uint32_t site) {
    if (status != nullptr && atomicCAS(status + kStatusCode, 0u, uint32_t(kDevTimeout)) == 0u)
        atomicExch(status + kStatusWhere, site);
}

// Wait for phase `parity` of `bar`; false (and status recorded) after the limit.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status, uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) {
            report_timeout(status, site);
            return false;
        }
    }
    return true;
}

}  // namespace tlb
