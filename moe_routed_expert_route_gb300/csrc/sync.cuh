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

// Arrive on a completion counter and wait until `target` CTAs have arrived:
// one thread per CTA polls one word. Bounded: on timeout records
// MOE_ERR_DEVICE_TIMEOUT, sets *abort and returns (results are then invalid),
// so a broken launch ends instead of hanging the GPU.
__device__ __forceinline__ void arrive_and_wait(unsigned* counter, unsigned target, int* status, int* abort) {
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

// Values exchanged between the CTAs of one launch carry a tag derived from the
// launch's sequence number in the upper 32 bits of one 64-bit word, so a reader
// can tell a value of this launch from a stale one without a separate barrier:
// it polls the data itself. 64-bit aligned accesses are single-copy atomic.
// The tag is a negative quiet-NaN bit pattern holding 22 bits of the sequence
// number: zeroed memory and ordinary float data never look like a current tag.
__device__ __forceinline__ unsigned seq_tag(unsigned seq) { return 0xFFC00000u | (seq & 0x3FFFFFu); }
__device__ __forceinline__ void st_tagged(uint64_t* p, float v, unsigned tag) {
    uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t* p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ bool tag_ok(uint64_t w, unsigned tag) { return (unsigned)(w >> 32) == tag; }
__device__ __forceinline__ float tag_val(uint64_t w) { return __uint_as_float((unsigned)w); }

// Reads n tagged values [i0, i0 + n*stride) of this launch into out[] (n is a
// compile-time bound, entries with i >= limit read as 0), polling until every
// value carries `tag`. Bounded: on timeout records MOE_ERR_DEVICE_TIMEOUT,
// sets *abort and returns what it has.
template <int N>
__device__ __forceinline__ void ld_tagged_all(const uint64_t* base, int i0, int stride, int limit,
                                              unsigned tag, float* out, int* status, int* abort) {
    bool ready[N];
#pragma unroll
    for (int q = 0; q < N; q++) {
        int i = i0 + q * stride;
        ready[q] = i >= limit;
        out[q] = 0.f;
    }
    long long t0 = clock64();
    while (true) {
        uint64_t w[N];
#pragma unroll
        for (int q = 0; q < N; q++)  // all loads in flight before the first is examined
            if (!ready[q]) w[q] = ld_tagged(base + i0 + q * stride);
        bool all = true;
#pragma unroll
        for (int q = 0; q < N; q++) {
            if (!ready[q]) {
                if (tag_ok(w[q], tag)) {
                    ready[q] = true;
                    out[q] = tag_val(w[q]);
                } else {
                    all = false;
                }
            }
        }
        if (all || *abort) break;
        if (clock64() - t0 > kSpinLimitCycles) {
            record_error(status, MOE_ERR_DEVICE_TIMEOUT);
            *abort = 1;
            break;
        }
    }
}

}  // namespace moe
