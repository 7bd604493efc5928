// Routed experts of the MoE block for decode-sized batches.
//
// Qiita "custom Metal gather_qmm", section 4: the routing indices are an input
// of the kernel and the expert id is used as a run-time index into the stacked
// weights, so experts nobody routed to are never fetched. Section 7: gate and
// up read the token's shared x, down reads each slot's own gated activation.
//
// Kernels (one launch each, chained with programmatic dependent launch):
//   prep_kernel      groups the (token, slot) assignments by expert and writes
//                    the fixed-point copy of x (only for moe_decode; in a whole
//                    layer the router kernel does both)
//   gateup_kernel    one warp per (distinct expert, output row n): the gate row
//                    and the up row are read once with 16-byte coalesced loads
//                    and applied to every token routed to that expert;
//                    h[t][r][n] = silu(g) * u
//   down_kernel      one warp per (token, output row d): the k down rows of the
//                    token's experts, combined with the routing weights in
//                    registers; y[t][d] and optionally x_next = x + y
//
// Dot products run on the integer pipe: a quantised weight block (int8, or
// int4 widened to 16*q by masking its nibbles into the top of each byte) times
// the 16-bit fixed-point activation block via dp4a, exact in int32, then one
// fp32 multiply by (weight scale * activation scale) per 16-byte chunk.
#include "dots.cuh"
#include "group.cuh"
#include "kernels.h"

namespace moe {

template <int QB>
struct Chunk {
    // bytes of codes per 16-byte chunk -> elements, and the chunk's block
    static constexpr int kElems = QB == 8 ? 16 : 32;
    static __device__ __forceinline__ int block(int c) { return QB == 8 ? (c >> 1) : c; }
    static constexpr float kScale = QB == 8 ? 1.0f : (1.0f / 16.0f);
};

// Plane dot of chunk c of a row against an activation's planes (global, L2).
template <int QB>
__device__ __forceinline__ int dot_chunk_global(const uint4 q, const int8_t* hi, const uint8_t* lo, int c) {
    if constexpr (QB == 8) {
        return dot_i8_chunk(q, ld_cg16(hi + 16 * c), ld_cg16(lo + 16 * c));
    } else {
        return dot_i4_chunk(q, ld_cg16(hi + 32 * c), ld_cg16(hi + 32 * c + 16), ld_cg16(lo + 32 * c),
                            ld_cg16(lo + 32 * c + 16));
    }
}
template <int QB>
__device__ __forceinline__ int dot_chunk_shared(const uint4 q, const int8_t* hi, const uint8_t* lo, int c) {
    if constexpr (QB == 8) {
        return dot_i8_chunk(q, *reinterpret_cast<const uint4*>(hi + 16 * c),
                            *reinterpret_cast<const uint4*>(lo + 16 * c));
    } else {
        const uint4* H = reinterpret_cast<const uint4*>(hi + 32 * c);
        const uint4* L = reinterpret_cast<const uint4*>(lo + 32 * c);
        return dot_i4_chunk(q, H[0], H[1], L[0], L[1]);
    }
}

// ------------------------------------------------------------------- prep
__global__ void __launch_bounds__(256) prep_kernel(PrepParams p) {
    extern __shared__ int s_mem[];
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0) {
        group_assignments(p.idx, p.T * p.k, p.E, p.hdr, p.grp_expert, p.grp_off, p.assign, s_mem);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = p.D / kBlk;
    for (int blk = (blockIdx.x - 1) * 8 + warp; blk < p.T * nb; blk += (gridDim.x - 1) * 8) {
        int t = blk / nb, b = blk - t * nb;
        size_t base = (size_t)t * p.D + b * kBlk;
        float v = p.x_bf16 ? ldcg_f32(reinterpret_cast<const __nv_bfloat16*>(p.x) + base + lane)
                           : ldcg_f32(reinterpret_cast<const float*>(p.x) + base + lane);
        fx_store_block(v, lane, p.qbits, p.xq_hi + base, p.xq_lo + base, p.xq_s + (size_t)t * nb + b);
    }
}

cudaError_t launch_prep(const PrepParams& p, cudaStream_t s, bool pdl) {
    int nblk = p.T * (p.D / kBlk);
    int grid = 1 + std::min(1024, (nblk + 7) / 8);
    return launch(prep_kernel, dim3(grid), dim3(256), sizeof(int) * (2 * p.E + 1), s, pdl, p);
}

// ---------------------------------------------------------------- gate/up
template <int QB, typename ST, int NCH>
__global__ void __launch_bounds__(256) gateup_kernel(ExpertParams p) {
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * 8;
    const int rowbytes = QB == 8 ? p.D : p.D / 2;
    const int nchunk = rowbytes / 16;
    const int nb = p.D / kBlk;
    const uint8_t* GQ = reinterpret_cast<const uint8_t*>(p.gate_q);
    const uint8_t* UQ = reinterpret_cast<const uint8_t*>(p.up_q);
    const ST* GS = reinterpret_cast<const ST*>(p.gate_s);
    const ST* US = reinterpret_cast<const ST*>(p.up_s);

    pdl_wait();
    pdl_trigger();
    for (int task = gwarp; task < p.max_groups * p.F; task += nwarps) {
        const int g = task / p.F;
        const int n = task - g * p.F;
        // the group count and the group's entries are fetched together; g is
        // below the workspace's group capacity, so the speculative reads stay
        // inside it
        const int ng = ld_cg_i32(&p.hdr->n_groups);
        const int e = ld_cg_i32(p.grp_expert + g);
        const int a0 = ld_cg_i32(p.grp_off + g), a1 = ld_cg_i32(p.grp_off + g + 1);
        const int asg0 = ld_cg_i32(p.assign + min(max(a0, 0), p.T * p.k - 1));
        if (g >= ng) break;
        const size_t row = (size_t)e * p.F + n;
        uint4 gv[NCH], uv[NCH];
        float gsc[NCH], usc[NCH];
#pragma unroll
        for (int j = 0; j < NCH; j++) {
            int c = j * 32 + lane;
            if (c < nchunk) {
                gv[j] = ld_stream16(GQ + row * rowbytes + 16 * c);
                uv[j] = ld_stream16(UQ + row * rowbytes + 16 * c);
                gsc[j] = to_f32(GS[row * nb + Chunk<QB>::block(c)]) * Chunk<QB>::kScale;
                usc[j] = to_f32(US[row * nb + Chunk<QB>::block(c)]) * Chunk<QB>::kScale;
            } else {
                gv[j] = uv[j] = make_uint4(0, 0, 0, 0);
                gsc[j] = usc[j] = 0.f;
            }
        }
        for (int a = a0; a < a1; a++) {
            const int asg = a == a0 ? asg0 : ld_cg_i32(p.assign + a);
            const int t = asg / p.k;
            const int8_t* xh = p.xq_hi + (size_t)t * p.D;
            const uint8_t* xl = p.xq_lo + (size_t)t * p.D;
            const float* xs = p.xq_s + (size_t)t * nb;
            float ga = 0.f, ua = 0.f;
#pragma unroll
            for (int j = 0; j < NCH; j++) {
                int c = j * 32 + lane;
                if (c < nchunk) {
                    float s = ld_cg_f32(xs + Chunk<QB>::block(c));
                    int ig, iu;
                    if constexpr (QB == 8) {
                        uint4 hi = ld_cg16(xh + 16 * c), lo = ld_cg16(xl + 16 * c);
                        ig = dot_i8_chunk(gv[j], hi, lo);
                        iu = dot_i8_chunk(uv[j], hi, lo);
                    } else {
                        uint4 h0 = ld_cg16(xh + 32 * c), h1 = ld_cg16(xh + 32 * c + 16);
                        uint4 l0 = ld_cg16(xl + 32 * c), l1 = ld_cg16(xl + 32 * c + 16);
                        ig = dot_i4_chunk(gv[j], h0, h1, l0, l1);
                        iu = dot_i4_chunk(uv[j], h0, h1, l0, l1);
                    }
                    ga = fmaf((float)ig, gsc[j] * s, ga);
                    ua = fmaf((float)iu, usc[j] * s, ua);
                }
            }
            ga = warp_sum(ga);
            ua = warp_sum(ua);
            if (lane == 0) p.h[(size_t)asg * p.F + n] = silu_mul(ga, ua);
        }
    }
}

// ------------------------------------------------------------------- down
constexpr int kConvBatch = 24;  // h blocks converted per warp per round trip

template <int QB, typename ST, int NLD>
__global__ void __launch_bounds__(256) down_kernel(ExpertParams p) {
    extern __shared__ __align__(16) unsigned char s_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nbd = (p.D + 7) / 8;
    const int t = blockIdx.x / nbd;
    const int d = (blockIdx.x - t * nbd) * 8 + warp;
    const int rowbytes = QB == 8 ? p.F : p.F / 2;
    const int nch = rowbytes / 16;
    const int total = p.k * nch;
    const int nbF = p.F / kBlk;
    int8_t* s_hi = reinterpret_cast<int8_t*>(s_raw);
    uint8_t* s_lo = s_raw + (size_t)p.k * p.F;
    float* s_sc = reinterpret_cast<float*>(s_raw + (size_t)2 * p.k * p.F);
    const uint8_t* DQ = reinterpret_cast<const uint8_t*>(p.down_q);
    const ST* DS = reinterpret_cast<const ST*>(p.down_s);

    // Weights first: they depend only on the routing, which is complete before
    // this grid can start (the previous kernel waited for it).
    uint4 v[NLD];
    float sc[NLD];
#pragma unroll
    for (int i = 0; i < NLD; i++) {
        int c = i * 32 + lane;
        v[i] = make_uint4(0, 0, 0, 0);
        sc[i] = 0.f;
        if (c < total && d < p.D) {
            int r = c / nch, cc = c - r * nch;
            int e = ld_cg_i32(p.idx + (size_t)t * p.k + r);
            if (e >= 0 && e < p.E) {
                size_t row = (size_t)e * p.D + d;
                v[i] = ld_stream16(DQ + row * rowbytes + 16 * cc);
                sc[i] = to_f32(DS[row * nbF + Chunk<QB>::block(cc)]) * Chunk<QB>::kScale;
            } else {
                record_error(&p.hdr->status, MOE_ERR_BAD_INDEX);
            }
        }
    }
    pdl_wait();
    pdl_trigger();

    // this token's gated activations, k slots x F, into fixed point (scale
    // folded with the slot's routing weight); the loads of a batch are all
    // issued before the first is used
    const int nblk = p.k * nbF;
    const float* ht = p.h + (size_t)t * p.k * p.F;
    for (int base = warp; base < nblk; base += 8 * kConvBatch) {
        float hv[kConvBatch], wr[kConvBatch];
#pragma unroll
        for (int i = 0; i < kConvBatch; i++) {
            int blk = base + 8 * i;
            hv[i] = blk < nblk ? ld_cg_f32(ht + (size_t)blk * kBlk + lane) : 0.f;
            wr[i] = blk < nblk ? ld_cg_f32(p.w + (size_t)t * p.k + blk / nbF) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kConvBatch; i++) {
            int blk = base + 8 * i;
            if (blk < nblk) {
                float m = warp_max(fabsf(hv[i]));
                Fx f = fx_of_blockmax(m);
                int X = fx_code(hv[i], f.mul);
                int pos = blk * kBlk + fx_pos(lane, QB);
                s_hi[pos] = (int8_t)(X >> 8);
                s_lo[pos] = (uint8_t)(X & 0xff);
                if (lane == 0) s_sc[blk] = f.scale * wr[i];
            }
        }
    }
    __syncthreads();
    if (d >= p.D) return;

    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < NLD; i++) {
        int c = i * 32 + lane;
        if (c < total) {
            int r = c / nch, cc = c - r * nch;
            int dot = dot_chunk_shared<QB>(v[i], s_hi + r * p.F, s_lo + r * p.F, cc);
            acc = fmaf((float)dot, sc[i] * s_sc[r * nbF + Chunk<QB>::block(cc)], acc);
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) {
        size_t o = (size_t)t * p.D + d;
        p.y[o] = acc;
        if (p.x_next) {
            if (p.x_bf16) {
                float xv = ldcg_f32(reinterpret_cast<const __nv_bfloat16*>(p.x) + o);
                reinterpret_cast<__nv_bfloat16*>(p.x_next)[o] = __float2bfloat16_rn(xv + acc);
            } else {
                float xv = ldcg_f32(reinterpret_cast<const float*>(p.x) + o);
                reinterpret_cast<float*>(p.x_next)[o] = xv + acc;
            }
        }
    }
}

// --------------------------------------------------------------- dispatch
static int chunks_per_lane(int chunks) { return (chunks + 31) / 32; }

static int down_nld(int k, int F, int qbits) {
    int nch = (qbits == 8 ? F : F / 2) / 16;
    int n = chunks_per_lane(k * nch);
    if (n <= 1) return 1;
    if (n <= 2) return 2;
    if (n <= 4) return 4;
    if (n <= 8) return 8;
    if (n <= 12) return 12;
    if (n <= 16) return 16;
    return 0;
}

static int gateup_nch(int D, int qbits) {
    int n = chunks_per_lane((qbits == 8 ? D : D / 2) / 16);
    if (n <= 1) return 1;
    if (n <= 2) return 2;
    if (n <= 4) return 4;
    if (n <= 8) return 8;
    return 0;
}

static size_t down_smem(int k, int F) { return (size_t)2 * k * F + sizeof(float) * k * (F / kBlk); }

bool experts_supported(int T, int E, int D, int F, int k, int qbits) {
    (void)T;
    (void)E;
    return down_nld(k, F, qbits) != 0 && gateup_nch(D, qbits) != 0 && down_smem(k, F) <= 160 * 1024;
}

template <int QB, typename ST, int NCH>
static cudaError_t launch_gateup_t(const ExpertParams& p, cudaStream_t s) {
    long ntask = (long)p.max_groups * p.F;
    long ctas = std::min<long>((ntask + 7) / 8, 152L * 16);
    return launch(gateup_kernel<QB, ST, NCH>, dim3((unsigned)std::max<long>(ctas, 1)), dim3(256), 0, s, true, p);
}
template <int QB, typename ST>
static cudaError_t launch_gateup_q(const ExpertParams& p, cudaStream_t s) {
    switch (gateup_nch(p.D, QB)) {
        case 1: return launch_gateup_t<QB, ST, 1>(p, s);
        case 2: return launch_gateup_t<QB, ST, 2>(p, s);
        case 4: return launch_gateup_t<QB, ST, 4>(p, s);
        default: return launch_gateup_t<QB, ST, 8>(p, s);
    }
}
template <int QB, typename ST, int NLD>
static cudaError_t launch_down_t(const ExpertParams& p, cudaStream_t s) {
    dim3 grid(p.T * ((p.D + 7) / 8));
    return launch(down_kernel<QB, ST, NLD>, grid, dim3(256), down_smem(p.k, p.F), s, true, p);
}
template <int QB, typename ST>
static cudaError_t launch_down_q(const ExpertParams& p, cudaStream_t s) {
    switch (down_nld(p.k, p.F, QB)) {
        case 1: return launch_down_t<QB, ST, 1>(p, s);
        case 2: return launch_down_t<QB, ST, 2>(p, s);
        case 4: return launch_down_t<QB, ST, 4>(p, s);
        case 8: return launch_down_t<QB, ST, 8>(p, s);
        case 12: return launch_down_t<QB, ST, 12>(p, s);
        default: return launch_down_t<QB, ST, 16>(p, s);
    }
}
template <int QB>
static cudaError_t launch_experts_q(const ExpertParams& p, cudaStream_t s) {
    cudaError_t e = p.s_f16 ? launch_gateup_q<QB, __half>(p, s) : launch_gateup_q<QB, float>(p, s);
    if (e != cudaSuccess) return e;
    return p.s_f16 ? launch_down_q<QB, __half>(p, s) : launch_down_q<QB, float>(p, s);
}

cudaError_t launch_experts(const ExpertParams& p, cudaStream_t s) {
    return p.qbits == 8 ? launch_experts_q<8>(p, s) : launch_experts_q<4>(p, s);
}

}  // namespace moe
