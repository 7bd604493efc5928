// mbarrier, bulk-copy (TMA) and inter-CTA exchange helpers (sm_90+ PTX), all waits bounded.
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

// Prefetch of `bytes` (multiple of 16, 16-byte aligned) of global memory into
// L2, without waiting and without a destination.
__device__ __forceinline__ void prefetch_l2(const void* src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
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
// if the phase did not complete within `limit` cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned phase, int* status,
                                          long long limit = kSpinLimitCycles) {
    long long t0 = clock64();
    while (!mbar_try_wait(bar, phase)) {
        if (clock64() - t0 > limit) {
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

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Values exchanged between the CTAs of one launch carry a tag derived from the
// launch's sequence number (the upper 32 bits of one 64-bit word, or a whole
// 32-bit flag word), so a reader can tell a value of this launch from a stale
// one by polling the data itself. 64-bit aligned accesses are single-copy
// atomic. A tag is never 0, so zeroed memory never carries a current tag, and
// for the first 2^22 sequence numbers it is a negative quiet-NaN bit pattern,
// which finite float data never is; tags repeat only after 2^32 launches.
__device__ __forceinline__ unsigned seq_tag(unsigned seq) {
    unsigned t = (seq + 1u) ^ 0xFFC00000u;
    return t ? t : 0xFFC00000u;
}
__device__ __forceinline__ void st_tagged(uint64_t* p, float v, unsigned tag) {
    uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t* p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
// A 32-bit payload (a float, or two 16-bit values) under a tag.
__device__ __forceinline__ void st_tagged_u32(uint64_t* p, uint32_t v, unsigned tag) {
    uint64_t w = ((uint64_t)tag << 32) | v;
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// Two consecutive tagged words (16-byte aligned); each is read single-copy atomically.
__device__ __forceinline__ void ld_tagged2(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ bool tag_ok(uint64_t w, unsigned tag) { return (unsigned)(w >> 32) == tag; }
__device__ __forceinline__ float tag_val(uint64_t w) { return __uint_as_float((unsigned)w); }

// Called by one whole warp: polls the n flag words flags[0..n) until every one
// holds `tag` (all loads of a round in flight before any is examined), then
// fences so that what the flags' writers stored before their release is
// visible. Bounded: on timeout records MOE_ERR_DEVICE_TIMEOUT and returns false.
__device__ __forceinline__ bool poll_flags(const unsigned* flags, int n, unsigned tag, long long limit,
                                           int* status) {
    const int lane = threadIdx.x & 31;
    const long long t0 = clock64();
    while (true) {
        bool all = true;
        for (int i = lane; i < n; i += 32) all &= ld_relaxed_u32(flags + i) == tag;
        if (__all_sync(0xffffffffu, all)) break;
        if (clock64() - t0 > limit) {
            if (lane == 0) record_error(status, MOE_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
    fence_acq_rel_gpu();
    return true;
}

}  // namespace moe
