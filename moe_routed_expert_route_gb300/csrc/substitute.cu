// Residency substitution of routed experts.
// gist.science "Which expert misses are worth waiting for?", method section:
// with only part of the experts resident, a missed expert is fetched when it is
// the router's first choice or its gate weight is >= 0.15, and otherwise
// replaced by a resident expert; the substituted gate mass m of a token is the
// sum of the normalised gate weights of its substituted experts. Fetch-all
// (threshold 0) and the first-choice rule (threshold +inf) are the same kernel.
//
// One warp per token. Lane l keeps the candidate keys of experts l, l+32, ...:
// resident experts that are not among the token's k routed ones, keyed by
// their fp32 probability; a replacement is the largest key (lower id on equal
// probability), which is then removed so it cannot be chosen twice.
#include "kernels.h"

namespace moe {

template <int NJ>
__global__ void __launch_bounds__(256) substitute_kernel(SubstituteParams p) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    pdl_wait();
    pdl_trigger();
    if (t >= p.T) return;
    const float* pt = p.probs + (size_t)t * p.E;
    unsigned key[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        int e = j * 32 + lane;
        key[j] = (e < p.E && p.resident[e]) ? __float_as_uint(ld_cg_f32(pt + e)) + 1u : 0u;
    }
    int my_e = lane < p.k ? ld_cg_i32(p.idx_in + (size_t)t * p.k + lane) : -1;
    float my_w = lane < p.k ? ld_cg_f32(p.w_in + (size_t)t * p.k + lane) : 0.f;
    for (int r = 0; r < p.k; r++) {
        int er = __shfl_sync(kFull, my_e, r);
#pragma unroll
        for (int j = 0; j < NJ; j++)
            if (j * 32 + lane == er) key[j] = 0u;
    }
    float mass = 0.f;
    for (int r = 0; r < p.k; r++) {
        int er = __shfl_sync(kFull, my_e, r);
        float wr = __shfl_sync(kFull, my_w, r);
        int out = er;
        uint8_t flag;
        if (er < 0 || er >= p.E) {
            flag = 1;  // an id outside [0, E) is passed through untouched, never dereferenced
        } else if (p.resident[er]) {
            flag = 0;
        } else if (r == 0 || wr >= p.threshold) {
            flag = 1;
        } else {
            unsigned bk = 0;
            int be = 0x7fffffff;
#pragma unroll
            for (int j = 0; j < NJ; j++)
                if (key[j] > bk) { bk = key[j]; be = j * 32 + lane; }
            unsigned mk = __reduce_max_sync(kFull, bk);
            if (mk == 0u) {
                flag = 3;
            } else {
                unsigned cand = (bk == mk) ? (unsigned)be : 0x7fffffffu;
                int we = (int)__reduce_min_sync(kFull, cand);
#pragma unroll
                for (int j = 0; j < NJ; j++)
                    if (j * 32 + lane == we) key[j] = 0u;
                out = we;
                flag = 2;
                mass += wr;
            }
        }
        if (lane == 0) {
            size_t o = (size_t)t * p.k + r;
            p.idx_out[o] = out;
            p.w_out[o] = wr;
            p.flag[o] = flag;
        }
    }
    if (lane == 0) p.mass[t] = mass;
}

cudaError_t launch_substitute(const SubstituteParams& p, cudaStream_t s) {
    dim3 grid((p.T + 7) / 8), block(256);
    if (p.E <= 32) return launch(substitute_kernel<1>, grid, block, 0, s, true, p);
    if (p.E <= 256) return launch(substitute_kernel<8>, grid, block, 0, s, true, p);
    if (p.E <= 512) return launch(substitute_kernel<16>, grid, block, 0, s, true, p);
    return launch(substitute_kernel<32>, grid, block, 0, s, true, p);
}

}  // namespace moe
