// mbarrier, bulk-copy (TMA) and grid-barrier helpers (sm_90+ PTX), all waits bounded.
#pragma once

#include "common.cuh"

namespace moe {

// Cycles a wait may spin before it gives up and reports MOE_ERR_DEVICE_TIMEOUT
// (about 30 ms at 2 GHz): far above any legitimate wait in one launch.
constexpr long long kSpinLimitCycles = 1LL << 26;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) whose completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned phase) {
    unsigned done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(phase)
        : "memory");
    return done != 0;
}

// Bounded wait on an mbarrier phase. Returns false (and records a timeout)
// if the phase did not complete within kSpinLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned phase, int* status) {
    long long t0 = clock64();
    while (!mbar_try_wait(bar, phase)) {
        if (clock64() - t0 > kSpinLimitCycles) {
            record_error(status, MOE_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier over a counter that only grows within a launch: barrier
// number b (1, 2, ...) completes when the counter reaches b * nblocks. All CTAs
// of the grid must be resident (one CTA per SM, grid <= SM count). The wait is
// bounded: on timeout the status word records MOE_ERR_DEVICE_TIMEOUT, `*abort`
// is set and the CTA goes on (its results are then not valid), so a broken
// launch ends instead of hanging the GPU.
__device__ __forceinline__ void grid_barrier(unsigned* counter, unsigned target, int* status, int* abort) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add(counter, 1u);
        if (!*abort) {
            long long t0 = clock64();
            while (ld_acquire_u32(counter) < target) {
                if (clock64() - t0 > kSpinLimitCycles) {
                    record_error(status, MOE_ERR_DEVICE_TIMEOUT);
                    *abort = 1;
                    break;
                }
            }
        }
    }
    __syncthreads();
}

// Last arrival of a launch: the CTA that brings the counter to `total` resets
// it to zero for the next launch (every CTA has passed every barrier by then).
__device__ __forceinline__ void grid_exit(unsigned* counter, unsigned total) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned prev = atomicAdd(counter, 1u);
        if (prev == total - 1) atomicExch(counter, 0u);
    }
}

}  // namespace moe
