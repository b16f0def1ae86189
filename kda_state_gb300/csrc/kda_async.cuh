// Asynchronous global -> shared copies for persistent kernels: an mbarrier
// counts the bytes of plain bulk copies (cp.async.bulk, no tensor map), and
// waits on it are bounded by %globaltimer so that a copy that never lands
// ends in an error status instead of a hang.
#pragma once

#include <stdint.h>

namespace kda {

constexpr uint64_t ASYNC_WAIT_NS = 2000000000ull;   // 2 s

__device__ __forceinline__ uint32_t shared_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void barrier_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival that also announces `bytes` of copies completing on the barrier.
__device__ __forceinline__ void barrier_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// One arrival with no copies (completes the phase of a count-1 barrier).
__device__ __forceinline__ void barrier_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Wait for the phase with the given parity; false after limit_ns.
__device__ __forceinline__ bool barrier_wait_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (global_timer() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ bool barrier_wait(uint32_t bar, uint32_t parity) {
    return barrier_wait_for(bar, parity, ASYNC_WAIT_NS);
}
// bytes (a multiple of 16; both addresses 16-byte aligned) from global to
// shared memory, completing on bar.
__device__ __forceinline__ void bulk_copy(void *dst_shared, const void *src_global, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            shared_addr(dst_shared)),
        "l"(reinterpret_cast<uint64_t>(src_global)), "r"(bytes), "r"(bar)
        : "memory");
}
// Ask for bytes (a multiple of 16) of global memory to be brought into L2,
// without waiting and without a destination in shared memory.
__device__ __forceinline__ void prefetch_l2(const void *src_global, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src_global)),
                 "r"(bytes)
                 : "memory");
}
// Order this thread's earlier generic-proxy accesses of shared memory before
// later async-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace kda
