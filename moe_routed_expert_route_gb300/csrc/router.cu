// Router of the MoE block: logits = x . Wr^T + bias, fp32 softmax, top-k.
// lilting.ch "observing the Qwen MoE router", section "hooking the router":
// gate (a linear map to E logits) -> softmax(precise) -> the k largest.
//
// One warp owns one expert row of Wr and computes its logit for every token;
// the row is loaded before the grid waits on the previous kernel (it does not
// depend on it), so the 1 MiB router read overlaps the previous layer's tail.
// The last CTA to finish (one atomic ticket per CTA) runs the softmax and top-k
// of every token, one warp per token, and -- when asked -- groups the
// assignments by expert for the expert kernels. The same kernel also writes
// the fixed-point copy of x that the expert kernels' integer dots consume.
#include "group.cuh"
#include "kernels.h"

namespace moe {

template <typename WT, typename XT, int NCH, int NJ>
__global__ void __launch_bounds__(256) router_kernel(RouterParams p) {
    extern __shared__ int s_mem[];
    __shared__ int s_last;
    __shared__ uint64_t s_tk[8][kTopkScratch];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x * 8 + warp;
    constexpr int EPC = 16 / sizeof(WT);  // weights per 16-byte chunk
    const int nchunk = p.D / EPC;
    const WT* W = reinterpret_cast<const WT*>(p.W);
    const XT* X = reinterpret_cast<const XT*>(p.x);

    uint4 wv[NCH];
#pragma unroll
    for (int j = 0; j < NCH; j++) {
        int c = j * 32 + lane;
        if (e < p.E && c < nchunk) wv[j] = ld_stream16(W + (size_t)e * p.D + (size_t)c * EPC);
        else wv[j] = make_uint4(0, 0, 0, 0);
    }
    pdl_trigger();
    pdl_wait();

    for (int t = 0; t < p.T; t++) {
        float acc = 0.f;
        const XT* xt = X + (size_t)t * p.D;
#pragma unroll
        for (int j = 0; j < NCH; j++) {
            int c = j * 32 + lane;
            if (c < nchunk) {
                const uint32_t* wq = reinterpret_cast<const uint32_t*>(&wv[j]);
                float xf[EPC];
                load_f32_cg<XT, EPC>(xt + c * EPC, xf);
#pragma unroll
                for (int i = 0; i < EPC; i++) {
                    float wf;
                    if constexpr (sizeof(WT) == 2) wf = (i & 1) ? bf16hi(wq[i >> 1]) : bf16lo(wq[i >> 1]);
                    else wf = __uint_as_float(wq[i]);
                    acc = fmaf(wf, xf[i], acc);
                }
            }
        }
        acc = warp_sum(acc);
        if (lane == 0 && e < p.E) p.logits[(size_t)t * p.E + e] = acc + (p.bias ? p.bias[e] : 0.f);
    }

    if (p.xq_hi) {
        const int nb = p.D / kBlk;
        for (int blk = blockIdx.x * 8 + warp; blk < p.T * nb; blk += gridDim.x * 8) {
            int t = blk / nb, b = blk - t * nb;
            float v = ldcg_f32(X + (size_t)t * p.D + b * kBlk + lane);
            size_t base = (size_t)t * p.D + b * kBlk;
            fx_store_block(v, lane, p.qbits, p.xq_hi + base, p.xq_lo + base,
                           p.xq_s + (size_t)t * nb + b);
        }
    }

    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned prev = atomicAdd(&p.hdr->done, 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    for (int t = warp; t < p.T; t += 8) {
        int sel_e;
        float sel_p;
        softmax_topk_warp<NJ>(p.logits + (size_t)t * p.E, p.E, p.k,
                              p.probs ? p.probs + (size_t)t * p.E : nullptr, lane, s_tk[warp], sel_e, sel_p);
        float norm = warp_sum(lane < p.k ? sel_p : 0.f);
        if (lane < p.k) {
            p.idx[(size_t)t * p.k + lane] = sel_e;
            p.w[(size_t)t * p.k + lane] = p.norm_topk ? sel_p / norm : sel_p;
        }
    }
    if (p.grp_expert) {
        __syncthreads();
        group_assignments(p.idx, p.T * p.k, p.E, p.hdr, p.grp_expert, p.grp_off, p.assign, s_mem);
    }
    if (threadIdx.x == 0) p.hdr->done = 0u;
}

template <typename WT, typename XT, int NCH>
static cudaError_t launch_router_nj(const RouterParams& p, cudaStream_t s, bool pdl) {
    dim3 grid((p.E + 7) / 8), block(256);
    size_t smem = p.grp_expert ? sizeof(int) * (2 * p.E + 1) : 0;
    switch (topk_nj(p.E, p.k)) {
        case 1: return launch(router_kernel<WT, XT, NCH, 1>, grid, block, smem, s, pdl, p);
        case 2: return launch(router_kernel<WT, XT, NCH, 2>, grid, block, smem, s, pdl, p);
        case 4: return launch(router_kernel<WT, XT, NCH, 4>, grid, block, smem, s, pdl, p);
        case 8: return launch(router_kernel<WT, XT, NCH, 8>, grid, block, smem, s, pdl, p);
        case 16: return launch(router_kernel<WT, XT, NCH, 16>, grid, block, smem, s, pdl, p);
        default: return launch(router_kernel<WT, XT, NCH, 32>, grid, block, smem, s, pdl, p);
    }
}

template <typename WT, typename XT>
static cudaError_t launch_router_nch(const RouterParams& p, cudaStream_t s, bool pdl) {
    int nchunk = p.D / (16 / (int)sizeof(WT));
    int nch = (nchunk + 31) / 32;
    if (nch <= 1) return launch_router_nj<WT, XT, 1>(p, s, pdl);
    if (nch <= 2) return launch_router_nj<WT, XT, 2>(p, s, pdl);
    if (nch <= 4) return launch_router_nj<WT, XT, 4>(p, s, pdl);
    if (nch <= 8) return launch_router_nj<WT, XT, 8>(p, s, pdl);
    return launch_router_nj<WT, XT, 16>(p, s, pdl);
}

cudaError_t launch_router(const RouterParams& p, bool w_bf16, bool x_bf16, cudaStream_t s,
                          bool pdl) {
    if (w_bf16 && x_bf16) return launch_router_nch<__nv_bfloat16, __nv_bfloat16>(p, s, pdl);
    if (w_bf16) return launch_router_nch<__nv_bfloat16, float>(p, s, pdl);
    if (x_bf16) return launch_router_nch<float, __nv_bfloat16>(p, s, pdl);
    return launch_router_nch<float, float>(p, s, pdl);
}

}  // namespace moe
