// Grouping of (token, slot) assignments by expert, and the per-token top-k.
#pragma once

#include "common.cuh"

namespace moe {

// Groups the n routing assignments idx[0..n) (assignment i = token i/k, slot
// i%k) by expert, inside ONE CTA:
//   cnt[e]          number of assignments routed to e
//   groups          the distinct experts in ascending id order:
//                   grp_expert[g], grp_off[g] .. grp_off[g+1] into `assign`
//   assign[p]       assignment ids, experts ascending, ascending i inside an
//                   expert (a stable counting sort)
// hdr->n_groups receives the number of distinct experts. Ids outside [0, E)
// are recorded as MOE_ERR_BAD_INDEX and left out. Needs 2*E+1 ints of shared
// memory at `s` and blockDim.x a multiple of 32. The order inside an expert is
// produced by warp 0 walking the assignments 32 at a time, so it does not
// depend on the order in which atomics land.
__device__ inline void group_assignments(const int32_t* __restrict__ idx, int n, int E,
                                         WsHeader* hdr, int32_t* __restrict__ grp_expert,
                                         int32_t* __restrict__ grp_off,
                                         int32_t* __restrict__ assign, int* s) {
    int* s_cnt = s;       // [E]
    int* s_off = s + E;   // [E + 1]
    const int tid = threadIdx.x, bs = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += bs) s_cnt[e] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += bs) {
        int e = idx[i];
        if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
        else record_error(&hdr->status, MOE_ERR_BAD_INDEX);
    }
    __syncthreads();
    if (warp == 0) {
        // each lane scans a contiguous segment of experts
        const int seg = (E + 31) / 32;
        const int e0 = min(E, lane * seg), e1 = min(E, e0 + seg);
        int csum = 0, gsum = 0;
        for (int e = e0; e < e1; e++) { csum += s_cnt[e]; gsum += s_cnt[e] > 0; }
        int cinc = csum, ginc = gsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int a = __shfl_up_sync(kFull, cinc, o), b = __shfl_up_sync(kFull, ginc, o);
            if (lane >= o) { cinc += a; ginc += b; }
        }
        int off = cinc - csum, g = ginc - gsum;
        for (int e = e0; e < e1; e++) {
            int c = s_cnt[e];
            s_off[e] = off;
            if (c > 0) { grp_expert[g] = e; grp_off[g] = off; g++; }
            off += c;
        }
        if (lane == 31) {
            hdr->n_groups = ginc;
            grp_off[ginc] = cinc;
            s_off[E] = cinc;
        }
        __syncwarp();
        // stable positions: rounds of 32 consecutive assignments
        const unsigned lt = (1u << lane) - 1u;
        for (int base = 0; base < n; base += 32) {
            int i = base + lane;
            int e = (i < n) ? idx[i] : -1;
            bool ok = (e >= 0 && e < E);
            int key = ok ? e : -2 - lane;  // unique key for lanes with nothing to place
            unsigned peers = __match_any_sync(kFull, key);
            int rank = __popc(peers & lt);
            int pos = ok ? s_off[e] + rank : 0;
            __syncwarp();
            if (ok) {
                assign[pos] = i;
                if (rank == 0) s_off[e] += __popc(peers);
            }
            __syncwarp();
        }
    }
    __syncthreads();
}

// Softmax and top-k of one token, by one warp, from logits already in
// registers: lane l holds the logits of experts l, l+32, ... (NJ per lane,
// NJ*32 >= E; entries e >= E are ignored). Probabilities are
// p_e = exp(l_e - max) / sum; the k largest are chosen largest first, equal
// fp32 values by lower expert id. Lanes r < k return (sel_e, sel_p) of rank r.
template <int NJ>
__device__ __forceinline__ void softmax_topk_regs(float (&p)[NJ], int E, int k, float* __restrict__ probs_t,
                                                  int lane, int& sel_e, float& sel_p) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < NJ; j++)
        if (j * 32 + lane < E) mx = fmaxf(mx, p[j]);
    mx = warp_max(mx);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        int e = j * 32 + lane;
        p[j] = (e < E) ? expf(p[j] - mx) : 0.f;
        s += p[j];
    }
    s = warp_sum(s);
    unsigned key[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        int e = j * 32 + lane;
        p[j] = p[j] / s;
        if (e < E && probs_t) probs_t[e] = p[j];
        key[j] = (e < E) ? __float_as_uint(p[j]) + 1u : 0u;  // p >= 0: bits are ordered
    }
    sel_e = -1;
    sel_p = 0.f;
    for (int r = 0; r < k; r++) {
        unsigned bk = 0;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < NJ; j++)
            if (key[j] > bk) { bk = key[j]; be = j * 32 + lane; }
        unsigned mk = __reduce_max_sync(kFull, bk);
        unsigned cand = (bk == mk && mk != 0u) ? (unsigned)be : 0x7fffffffu;
        unsigned we = __reduce_min_sync(kFull, cand);
        if (lane == r) { sel_e = (int)we; sel_p = __uint_as_float(mk - 1u); }
#pragma unroll
        for (int j = 0; j < NJ; j++)
            if (j * 32 + lane == (int)we) key[j] = 0u;
    }
}

// The same, reading the logits (written by an earlier kernel) through L2.
template <int NJ>
__device__ __forceinline__ void softmax_topk_warp(const float* __restrict__ logits_t, int E, int k,
                                                  float* __restrict__ probs_t, int lane,
                                                  int& sel_e, float& sel_p) {
    float p[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        int e = j * 32 + lane;
        p[j] = (e < E) ? ld_cg_f32(logits_t + e) : -INFINITY;
    }
    softmax_topk_regs<NJ>(p, E, k, probs_t, lane, sel_e, sel_p);
}

}  // namespace moe
