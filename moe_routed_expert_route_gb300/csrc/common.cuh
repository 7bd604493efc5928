// Device helpers shared by the routed-expert MoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_route.h"

namespace moe {

constexpr int kBlk = 32;           // quantisation block along the input dimension
constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------------------ workspace header
// The first 256 bytes of every workspace: device status word, the router's
// "CTAs finished" counter, the number of distinct routed experts, the launch
// sequence number that tags values exchanged between the CTAs of the
// persistent layer kernel, and the limit of every bounded device wait.
struct WsHeader {
    int status;
    unsigned int done;
    int n_groups;
    unsigned int bar;  // unused, zero
    unsigned int seq;  // launch sequence number of the persistent layer kernel
    unsigned int pad0[3];
    unsigned long long wait_limit;  // clock64 cycles a device wait may spin; 0 = default
    int pad[54];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

__device__ __forceinline__ void record_error(int* status, int code) {
    atomicCAS(status, 0, code);
}

// ------------------------------------------------ programmatic dependent launch
// wait: block until the grids this one depends on have completed and their
// memory is visible. trigger: allow the next grid in the stream to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// --------------------------------------------------------------- loads/stores
// Streaming 16-byte load of weights that are read once per call: skip L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// 16-byte load through L2 only (data written earlier by another CTA/kernel).
__device__ __forceinline__ uint4 ld_cg16(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_cg_f32(const float* p) { return __ldcg(p); }
// read-only (non-coherent) loads of data no kernel writes during the launch
template <typename T>
__device__ __forceinline__ uint4 ld_nc16(const T* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ float ldg_nc(const float* p) { return __ldg(p); }
__device__ __forceinline__ __half ldg_nc(const __half* p) { return __ldg(p); }
__device__ __forceinline__ int ld_cg_i32(const int* p) { return __ldcg(p); }

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One element written by an earlier kernel, read through L2.
__device__ __forceinline__ float ldcg_f32(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float ldcg_f32(const __nv_bfloat16* p) {
    unsigned short u = __ldcg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float((uint32_t)u << 16);
}

// N consecutive elements (16-byte aligned start) written by an earlier kernel,
// read through L2 and widened to fp32.
template <typename T, int N>
__device__ __forceinline__ void load_f32_cg(const T* p, float* out) {
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            uint4 v = ld_cg16(p + i);
            out[i] = __uint_as_float(v.x);
            if (i + 1 < N) out[i + 1] = __uint_as_float(v.y);
            if (i + 2 < N) out[i + 2] = __uint_as_float(v.z);
            if (i + 3 < N) out[i + 3] = __uint_as_float(v.w);
        }
    } else if constexpr (N % 8 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 8) {
            uint4 v = ld_cg16(p + i);
            const uint32_t* u = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
            for (int q = 0; q < 8; q++) out[i + q] = (q & 1) ? bf16hi(u[q >> 1]) : bf16lo(u[q >> 1]);
        }
    } else {
        static_assert(N == 4, "bf16 loads of 4 or a multiple of 8 elements");
        uint2 v = __ldcg(reinterpret_cast<const uint2*>(p));  // 8-byte aligned
        out[0] = bf16lo(v.x);
        out[1] = bf16hi(v.x);
        out[2] = bf16lo(v.y);
        out[3] = bf16hi(v.y);
    }
}

// --------------------------------------------------------------- integer dots
// d = c + sum_i a.byte[i] * b.byte[i]; a signed, b signed / unsigned.
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ------------------------------------------------------ fixed-point activations
// An activation vector is handed to the integer dot products as 16-bit fixed
// point with one power-of-two scale per block of 32 elements:
//   X_k = round(v_k * 2^(15 - e)),  |X_k| <= 32767,  v_k ~= X_k * 2^(e - 15)
// where 2^e is the smallest power of two above the block's max |v|. X is split
// into a signed high byte and an unsigned low byte (X = 256*hi + lo), so that
// sum_k q_k * X_k = 256 * dp4a(q, hi) + dp4a(q, lo) exactly in int32. A bf16
// value within 2^8 of the block max is represented exactly; the conversion
// error of any element is at most 2^(e-16). Blocks whose max |v| is below 2^-100
// (or zero) are stored as zero.
struct Fx {
    float mul;    // 2^(15 - e), 0 for a zero block
    float scale;  // 2^(e - 15), 0 for a zero block
};

__device__ __forceinline__ Fx fx_of_blockmax(float m) {
    Fx f;
    int bits = __float_as_int(m);
    int be = (bits >> 23) & 0xff;  // m in [2^(be-127), 2^(be-126))
    if (!(m >= 0x1p-100f) || be == 0xff) {
        f.mul = 0.f;
        f.scale = 0.f;
        return f;
    }
    int e = be - 126;  // m < 2^e
    f.mul = __int_as_float((127 + 15 - e) << 23);
    f.scale = __int_as_float((127 + e - 15) << 23);
    return f;
}

__device__ __forceinline__ int fx_code(float v, float mul) {
    int X = __float2int_rn(v * mul);
    return max(-32767, min(32767, X));
}

// Position of element k inside a block's plane. int8 codes use the natural
// order. int4 codes are consumed 8 at a time from one 32-bit word, even
// elements (low nibbles) and odd elements (high nibbles) separately, so their
// plane stores each group of 8 as [k0 k2 k4 k6 k1 k3 k5 k7].
__device__ __forceinline__ int fx_pos(int k, int qbits) {
    if (qbits == 8) return k;
    return (k & ~7) | ((k & 1) << 2) | ((k & 7) >> 1);
}

// Warp-wide reductions.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Quantise one block of 32 activations held one per lane and store it:
// hi/lo planes at [plane_off + fx_pos(lane)], scale at *scale_out (lane 0).
__device__ __forceinline__ void fx_store_block(float v, int lane, int qbits, int8_t* hi,
                                               uint8_t* lo, float* scale_out) {
    float m = warp_max(fabsf(v));
    Fx f = fx_of_blockmax(m);
    int X = fx_code(v, f.mul);
    int p = fx_pos(lane, qbits);
    hi[p] = (int8_t)(X >> 8);
    lo[p] = (uint8_t)(X & 0xff);
    if (lane == 0) *scale_out = f.scale;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

}  // namespace moe
