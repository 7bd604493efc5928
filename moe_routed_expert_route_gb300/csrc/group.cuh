// Grouping of (token, slot) assignments by expert, and the per-token top-k.
#pragma once

#include "common.cuh"

namespace moe {

// Values per lane for the one-warp top-k: a power of two with NJ*32 >= E and NJ >= k.
inline int topk_nj(int E, int k) {
    int need = (E + 31) / 32 > k ? (E + 31) / 32 : k;
    int nj = 1;
    while (nj < need) nj <<= 1;
    return nj;
}

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

// In-register bitonic networks on N (a power of two) unsigned 64-bit values,
// largest first. All indices are compile-time constants.
__device__ __forceinline__ void cas_desc(uint64_t& a, uint64_t& b) {
    uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
    a = hi;
    b = lo;
}
template <int N>
__device__ __forceinline__ void bitonic_merge_desc(uint64_t (&v)[N]) {
#pragma unroll
    for (int stride = N / 2; stride > 0; stride >>= 1)
#pragma unroll
        for (int i = 0; i < N; i++)
            if ((i & stride) == 0) cas_desc(v[i], v[i + stride]);
}
template <int N>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t (&v)[N]) {
#pragma unroll
    for (int size = 2; size <= N; size <<= 1)
#pragma unroll
        for (int stride = size / 2; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < N; i++) {
                const int j = i + stride;
                if ((i & stride) == 0) {
                    if ((i & size) == 0) cas_desc(v[i], v[j]);   // descending run
                    else cas_desc(v[j], v[i]);                   // ascending run
                }
            }
}

// The same networks on fp32 values (largest first).
template <int N>
__device__ __forceinline__ void bitonic_merge_desc_f(float (&v)[N]) {
#pragma unroll
    for (int stride = N / 2; stride > 0; stride >>= 1)
#pragma unroll
        for (int i = 0; i < N; i++)
            if ((i & stride) == 0) {
                const float hi = fmaxf(v[i], v[i + stride]), lo = fminf(v[i], v[i + stride]);
                v[i] = hi;
                v[i + stride] = lo;
            }
}
template <int N>
__device__ __forceinline__ void bitonic_sort_desc_f(float (&v)[N]) {
#pragma unroll
    for (int size = 2; size <= N; size <<= 1)
#pragma unroll
        for (int stride = size / 2; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < N; i++) {
                const int j = i + stride;
                if ((i & stride) == 0) {
                    const float hi = fmaxf(v[i], v[j]), lo = fminf(v[i], v[j]);
                    if ((i & size) == 0) { v[i] = hi; v[j] = lo; }   // descending run
                    else { v[i] = lo; v[j] = hi; }                   // ascending run
                }
            }
}

// Scratch of softmax_topk_regs: 2 * 32 keys per warp, warp-private.
constexpr int kTopkScratch = 64;

// Softmax and top-k of one token, by one warp, from logits already in
// registers: lane l holds the logits of experts l, l+32, ... (NJ per lane, a
// power of two, NJ*32 >= E, NJ >= k; entries e >= E are ignored).
// Probabilities are p_e = exp(l_e - max) * (1 / sum); the k largest are chosen
// largest first, equal fp32 values by lower expert id. Lanes r < k return
// (sel_e, sel_p) of rank r. `scratch` holds kTopkScratch 64-bit words of
// shared memory private to the warp.
//
// The selection works in two passes so that the long networks run on 32-bit
// values: the k-th largest logit l_k is found first (a per-lane sort and a
// butterfly that keeps the NJ largest of each union; its first entry is also
// the max the softmax needs). p is a non-decreasing function of l, so the k-th
// largest p is p* = p(l_k), read from an expert whose logit is l_k; the chosen
// experts are then every e with p_e > p* and, of those with p_e == p*, the
// lowest ids up to k. Only those k are ranked, by (p desc, id asc).
template <int NJ>
__device__ __forceinline__ void softmax_topk_regs(float (&p)[NJ], int E, int k, float* __restrict__ probs_t,
                                                  int lane, uint64_t* scratch, int& sel_e, float& sel_p) {
    float t[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) t[j] = (j * 32 + lane < E) ? p[j] : -INFINITY;
    bitonic_sort_desc_f<NJ>(t);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float b[NJ];
#pragma unroll
        for (int i = 0; i < NJ; i++) b[i] = __shfl_xor_sync(kFull, t[i], o);
#pragma unroll
        for (int i = 0; i < NJ; i++) t[i] = fmaxf(t[i], b[NJ - 1 - i]);
        bitonic_merge_desc_f<NJ>(t);
    }
    const float mx = t[0];
    float lk = t[0];
#pragma unroll
    for (int i = 0; i < NJ; i++)
        if (i == k - 1) lk = t[i];
    unsigned at_lk[NJ];  // which lanes hold an expert whose logit is l_k
#pragma unroll
    for (int j = 0; j < NJ; j++) at_lk[j] = __ballot_sync(kFull, j * 32 + lane < E && p[j] == lk);

    float s = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        int e = j * 32 + lane;
        p[j] = (e < E) ? expf(p[j] - mx) : 0.f;
        s += p[j];
    }
    s = warp_sum(s);
    const float inv_s = 1.0f / s;
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        int e = j * 32 + lane;
        p[j] = p[j] * inv_s;
        if (e < E && probs_t) probs_t[e] = p[j];
    }
    float pk = 0.f;
    bool found = false;
#pragma unroll
    for (int j = 0; j < NJ; j++)  // warp-uniform
        if (!found && at_lk[j]) {
            pk = __shfl_sync(kFull, p[j], __ffs(at_lk[j]) - 1);
            found = true;
        }

    // the chosen set, written in id order to scratch[0..k)
    const unsigned lt = (1u << lane) - 1u;
    int n_gt = 0;
    unsigned eqm[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        const bool valid = j * 32 + lane < E;
        n_gt += __popc(__ballot_sync(kFull, valid && p[j] > pk));
        eqm[j] = __ballot_sync(kFull, valid && p[j] == pk);
    }
    const int need = k - n_gt;  // >= 1 when the logits are finite
    int eq_before = 0, pos = 0;
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        const int e = j * 32 + lane;
        const bool valid = e < E;
        const bool take = valid && (p[j] > pk || (p[j] == pk && eq_before + __popc(eqm[j] & lt) < need));
        eq_before += __popc(eqm[j]);
        const unsigned tm = __ballot_sync(kFull, take);
        const int at = pos + __popc(tm & lt);
        // order key: fp32 bits + 1 of p >= 0 in the high word, ~id in the low
        // word: one unsigned comparison ranks "larger p first, lower id on equal p"
        if (take && at < k)
            scratch[at] = ((uint64_t)(__float_as_uint(p[j]) + 1u) << 32) | (uint64_t)(0xffffffffu - (unsigned)e);
        pos += __popc(tm);
    }
    __syncwarp();
    const int nsel = pos < k ? pos : k;
    uint64_t mine = 0;
    int rank = 0;
    if (lane < nsel) {
        mine = scratch[lane];
        for (int i = 0; i < nsel; i++) rank += scratch[i] > mine ? 1 : 0;
    }
    __syncwarp();
    if (lane < nsel) scratch[32 + rank] = mine;
    __syncwarp();
    sel_e = -1;
    sel_p = 0.f;
    if (lane < nsel) {
        const uint64_t v = scratch[32 + lane];
        sel_e = (int)(0xffffffffu - (unsigned)v);
        sel_p = __uint_as_float((unsigned)(v >> 32) - 1u);
    }
    __syncwarp();
}

// The same, reading the logits (written by an earlier kernel) through L2.
template <int NJ>
__device__ __forceinline__ void softmax_topk_warp(const float* __restrict__ logits_t, int E, int k,
                                                  float* __restrict__ probs_t, int lane, uint64_t* scratch,
                                                  int& sel_e, float& sel_p) {
    float p[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        int e = j * 32 + lane;
        p[j] = (e < E) ? ld_cg_f32(logits_t + e) : -INFINITY;
    }
    softmax_topk_regs<NJ>(p, E, k, probs_t, lane, scratch, sel_e, sel_p);
}

}  // namespace moe
