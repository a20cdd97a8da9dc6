// Tensor Memory Accelerator (TMA) loads, bulk copies and mbarriers for sm_103a, as
// inline PTX. Every wait on an mbarrier is bounded (about one second of %globaltimer);
// a caller that sees a timeout records an error code and leaves the kernel.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace wt {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s, the default limit
constexpr int kErrTmaTimeout = 1;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialization visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// asynchronous-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Same for global memory (generic stores later read by a TMA load).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Every kernel keeps its mbarriers at the start of dynamic shared memory (at most 32 of
// them). The thread that issues a CTA's copies keeps one mask in a register for the drain
// below: bit b flips with every phase it opens on barrier b, so it holds the parity of the
// number of phases issued there.
struct Issued {
    uint32_t par = 0;
};

__device__ __forceinline__ uint64_t* mbar_region() {
    extern __shared__ __align__(128) float4 smem_f4[];
    return reinterpret_cast<uint64_t*>(smem_f4);
}

// arrive.expect_tx on `bar` (one of the region's barriers) that also records the phase it
// opens in `iss`. Only the thread that issues a CTA's copies calls it.
__device__ __forceinline__ void mbar_expect_tx_noted(uint64_t* bar, uint32_t bytes, Issued& iss) {
    iss.par ^= 1u << (uint32_t)(bar - mbar_region());
    mbar_arrive_expect_tx(bar, bytes);
}

// After a timed-out wait, before the CTA leaves: wait, at most `limit_ns` in all, until
// the last phase issued on every barrier of `mask` (the initialized barriers that copies
// complete on) has completed, so that no copy lands in shared memory after the CTA is
// gone. Each barrier has at most one phase outstanding (a copy is issued on it only after
// its previous phase was waited for), and the last issued phase's parity is the opposite
// of the issue-count parity; on a barrier that never had a phase issued that test passes
// at once. Returns false if the limit ran out.
__device__ __forceinline__ bool mbar_drain_issued(const Issued& iss, uint32_t mask,
                                                  unsigned long long limit_ns);

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
// Coordinates are in elements; c0 * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the same phase (test_wait returns at once; try_wait may first
// suspend the thread for a while).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete; false once `limit_ns`
// nanoseconds have passed without it. A limit shorter than the default (only a test sets
// one) is counted in SM clock cycles, checked before every non-suspending probe:
// %globaltimer advances in steps of up to a microsecond and try_wait may suspend the
// thread for a while, either of which could outlast a short limit and hide it. At SM clocks
// of 1 GHz or more, that many cycles last no longer than that many nanoseconds; a limit
// shorter than one clock64 read gives up before the first probe, whether or not the copy
// has landed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
    if (limit_ns < kWaitLimitNs) {
        const long long c0 = clock64();
        while ((unsigned long long)(clock64() - c0) < limit_ns)
            if (mbar_test_wait(bar, parity)) return true;
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ bool mbar_drain_issued(const Issued& iss, uint32_t mask,
                                                  unsigned long long limit_ns) {
    uint64_t* base = mbar_region();
    const unsigned long long t0 = globaltimer_ns();
    for (int b = 0; b < 32; ++b) {
        if (((mask >> b) & 1u) == 0) continue;
        const uint32_t last = ((iss.par >> b) & 1u) ^ 1u;
        while (!mbar_try_wait(base + b, last))
            if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// One arrival on `bar` (release semantics: this thread's earlier shared-memory accesses are
// ordered before a waiter's acquire).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bulk copy of `bytes` contiguous bytes from global to shared memory, completing on `bar`
// (both addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

}  // namespace wt
