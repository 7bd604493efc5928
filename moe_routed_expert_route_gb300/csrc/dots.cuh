// Integer dot products of quantised weight chunks with fixed-point activation
// planes (see fx_* in common.cuh for the activation format).
#pragma once

#include "common.cuh"

namespace moe {

// 16 int8 codes (one 16-byte chunk) against the matching 16 plane bytes.
__device__ __forceinline__ int dot_i8_chunk(const uint4 q, const uint4 hi, const uint4 lo) {
    int h = dp4a_ss(q.x, hi.x, 0);
    h = dp4a_ss(q.y, hi.y, h);
    h = dp4a_ss(q.z, hi.z, h);
    h = dp4a_ss(q.w, hi.w, h);
    int l = dp4a_su(q.x, lo.x, 0);
    l = dp4a_su(q.y, lo.y, l);
    l = dp4a_su(q.z, lo.z, l);
    l = dp4a_su(q.w, lo.w, l);
    return h * 256 + l;
}

// 32 int4 codes (one 16-byte chunk = one quantisation block) against the 32
// plane bytes of that block, returning 16 * sum(q * X): each word's low
// nibbles (even elements) and high nibbles (odd elements) are moved to the top
// of their bytes, where a two's complement nibble reads as 16 * its value.
__device__ __forceinline__ int dot_i4_word(uint32_t w, uint32_t he, uint32_t ho, uint32_t le,
                                           uint32_t lo, int& h, int& l) {
    uint32_t ev = (w << 4) & 0xF0F0F0F0u;
    uint32_t od = w & 0xF0F0F0F0u;
    h = dp4a_ss(ev, he, h);
    h = dp4a_ss(od, ho, h);
    l = dp4a_su(ev, le, l);
    l = dp4a_su(od, lo, l);
    return 0;
}
__device__ __forceinline__ int dot_i4_chunk(const uint4 q, const uint4 h0, const uint4 h1,
                                            const uint4 l0, const uint4 l1) {
    int h = 0, l = 0;
    dot_i4_word(q.x, h0.x, h0.y, l0.x, l0.y, h, l);
    dot_i4_word(q.y, h0.z, h0.w, l0.z, l0.w, h, l);
    dot_i4_word(q.z, h1.x, h1.y, l1.x, l1.y, h, l);
    dot_i4_word(q.w, h1.z, h1.w, l1.z, l1.w, h, l);
    return h * 256 + l;
}

}  // namespace moe
