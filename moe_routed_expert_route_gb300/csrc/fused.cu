// One whole MoE layer for one token in ONE persistent launch (decode; a batch
// of up to three tokens is run as one launch per token).
//
// lilting.ch "observing the Qwen MoE router" (section "hooking the router"):
// router logits -> fp32 softmax -> top-k. Qiita "custom Metal gather_qmm"
// (sections 4 and 7): only the k routed experts' rows are read, gate and up
// share x, down takes each slot's own activation, and the slots are combined
// with the routing weights.
//
// Grid = one CTA of 16 warps per SM, all resident. The CTAs exchange two small
// vectors through L2: the logits are tagged with the launch's sequence number
// so that readers poll the data itself instead of meeting at a grid barrier:
//   0  before waiting on the previous launch: each CTA loads its slice of the
//      router weights (1-4 experts' rows) into registers
//   1  x -> shared memory; the CTA's logits -> workspace (tagged)
//   2  warp 0 of every CTA polls all E logits and runs the softmax + top-k
//      (no second exchange is needed to learn the routing); the 12 warps that
//      do not share warp 0's scheduler turn x into 16-bit fixed-point planes
//      meanwhile
//   3  one thread starts bulk (TMA) copies of this CTA's rows of the k down
//      matrices into shared memory while the 16 warps stream this CTA's share
//      of the k*F gate/up row pairs from HBM (two row pairs in flight per
//      warp) and write h = silu(g)*u to the workspace; the CTA then arrives on
//      a completion counter (polling ~150 KB of tagged activations from every
//      CTA would flood L2 while other CTAs still stream)
//   4  each warp owns one slot: it reads that slot's activations into
//      registers as 16-bit fixed point and dots them (integer dp4a) against the
//      staged down rows of its share of the CTA's rows; the CTA combines the k
//      slots in slot order,
//      y[d] = sum_r w[r] * o_r[d], and writes x_next = x + y.
// Without a router (moe_decode) phases 0-2 are replaced by reading idx/w.
#include "dots.cuh"
#include "group.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace moe {

constexpr int kFThreads = 512;
constexpr int kFWarps = 16;
constexpr int kNRC = 2;  // router 16-byte chunks per lane
constexpr int kNCH = 4;  // gate/up 16-byte chunks per lane
constexpr int kRU = 4;   // down rows reduced together

struct FusedLayout {
    size_t x, xhi, xlo, xs, dq, ds, part, total;
};

__host__ __device__ inline size_t fl_align(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline FusedLayout fused_layout(int D, int F, int k, int qbits, int s_bytes, int rows) {
    FusedLayout L;
    size_t o = 0;
    const size_t rowF = qbits == 8 ? F : F / 2;
    L.x = o;    o = fl_align(o + sizeof(float) * D, 16);
    L.xhi = o;  o = fl_align(o + D, 16);
    L.xlo = o;  o = fl_align(o + D, 16);
    L.xs = o;   o = fl_align(o + sizeof(float) * (D / kBlk), 16);
    L.dq = o;   o = fl_align(o + (size_t)k * rows * rowF, 16);
    L.ds = o;   o = fl_align(o + (size_t)k * rows * (F / kBlk) * s_bytes, 16);
    L.part = o; o = fl_align(o + sizeof(float) * (size_t)k * rows, 16);
    L.total = o;
    return L;
}

template <int QB, typename ST>
struct RowPair {
    uint4 g[kNCH], u[kNCH];
    ST gs[kNCH], us[kNCH];  // widened where used, so no load is waited for early
};

// Fixed-point conversion of NB blocks of 32 values held one per lane, the
// NB max-reductions interleaved so their shuffles overlap.
template <int NB>
__device__ __forceinline__ void fx_store_blocks(const float (&v)[NB], const int (&blk)[NB], int nblk, int lane,
                                                int qbits, int8_t* hi, uint8_t* lo, float* scale) {
    float m[NB];
#pragma unroll
    for (int i = 0; i < NB; i++) m[i] = fabsf(v[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int i = 0; i < NB; i++) m[i] = fmaxf(m[i], __shfl_xor_sync(kFull, m[i], o));
#pragma unroll
    for (int i = 0; i < NB; i++) {
        if (blk[i] < nblk) {
            Fx f = fx_of_blockmax(m[i]);
            int X = fx_code(v[i], f.mul);
            int pos = blk[i] * kBlk + fx_pos(lane, qbits);
            hi[pos] = (int8_t)(X >> 8);
            lo[pos] = (uint8_t)(X & 0xff);
            if (lane == 0) scale[blk[i]] = f.scale;
        }
    }
}

template <int QB, typename ST, typename XT, int NJ>
__global__ void __launch_bounds__(kFThreads, 1) fused_layer_kernel(FusedParams p) {
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ float s_rpart[kFWarps];
    __shared__ int s_idx[32];
    __shared__ float s_w[32];
    __shared__ int s_abort;
    __shared__ unsigned s_seq;
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ uint64_t s_tk[kTopkScratch];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int D = p.D, F = p.F, k = p.k;
    const int nb = D / kBlk, nbF = F / kBlk;
    const int rowD = QB == 8 ? D : D / 2;    // bytes of a gate/up row
    const int rowF = QB == 8 ? F : F / 2;    // bytes of a down row
    const FusedLayout L = fused_layout(D, F, k, QB, sizeof(ST), p.rows);
    float* s_x = reinterpret_cast<float*>(sm + L.x);
    int8_t* s_xhi = reinterpret_cast<int8_t*>(sm + L.xhi);
    uint8_t* s_xlo = sm + L.xlo;
    float* s_xs = reinterpret_cast<float*>(sm + L.xs);
    uint8_t* s_dq = sm + L.dq;
    ST* s_ds = reinterpret_cast<ST*>(sm + L.ds);
    float* s_part = reinterpret_cast<float*>(sm + L.part);
    int* status = &p.hdr->status;

    // ---------------------------------------------------------- phase 0
    if (tid == 0) {
        s_abort = 0;
        mbar_init(&s_bar, 1);
        fence_barrier_init();
    }
    const XT* Wr = reinterpret_cast<const XT*>(p.W);
    constexpr int EPC = 16 / sizeof(XT);
    const int e_begin = (int)((long)c * p.E / G), e_end = (int)((long)(c + 1) * p.E / G);
    const int nseg = p.router_nseg;
    const int rj = warp / nseg, rs = warp - rj * nseg;
    const int re = e_begin + rj;
    const int seg = D / nseg;
    const bool rvalid = p.has_router && re < e_end;
    uint4 wr[kNRC];
#pragma unroll
    for (int i = 0; i < kNRC; i++) {
        int ci = i * 32 + lane;
        wr[i] = make_uint4(0, 0, 0, 0);
        if (rvalid && ci * EPC < seg) wr[i] = ld_stream16(Wr + (size_t)re * D + rs * seg + ci * EPC);
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    // the previous launch on this workspace has completed: its sequence
    // number increment is visible
    if (tid == 0) {
        s_seq = *reinterpret_cast<volatile unsigned*>(&p.hdr->seq);
        if (c == 0) p.hdr->hcount[(s_seq + 1) & 1] = 0u;  // the next launch's counter
    }

    // ---------------------------------------------------------- phase 1
    const XT* X = reinterpret_cast<const XT*>(p.x);
    for (int i = tid; i < D; i += kFThreads) s_x[i] = ldcg_f32(X + i);
    __syncthreads();
    const unsigned tag = seq_tag(s_seq);

    // x -> fixed-point planes. With a router, warp 0 selects the experts
    // meanwhile and the conversion runs on the 12 warps that do not share its
    // scheduler (warps w with w % 4 != 0), so the selection is not slowed.
    auto convert_x = [&](bool routing) {
        const int nw = routing ? kFWarps - kFWarps / 4 : kFWarps;
        const int wi = routing ? warp - (warp >> 2) - 1 : warp;
        for (int b0 = wi; b0 < nb; b0 += nw * 4) {
            float v[4];
            int blk[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                blk[i] = b0 + nw * i;
                v[i] = blk[i] < nb ? s_x[blk[i] * kBlk + lane] : 0.f;
            }
            fx_store_blocks<4>(v, blk, nb, lane, QB, s_xhi, s_xlo, s_xs);
        }
    };

    if (p.has_router) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < kNRC; i++) {
            int ci = i * 32 + lane;
            if (rvalid && ci * EPC < seg) {
                const float* xs = s_x + rs * seg + ci * EPC;
                const uint32_t* wq = reinterpret_cast<const uint32_t*>(&wr[i]);
#pragma unroll
                for (int q = 0; q < EPC; q++) {
                    float wf;
                    if constexpr (sizeof(XT) == 2) wf = (q & 1) ? bf16hi(wq[q >> 1]) : bf16lo(wq[q >> 1]);
                    else wf = __uint_as_float(wq[q]);
                    acc = fmaf(wf, xs[q], acc);
                }
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) s_rpart[warp] = acc;
        __syncthreads();
        if (tid < e_end - e_begin) {
            float l = 0.f;
            for (int s = 0; s < nseg; s++) l += s_rpart[tid * nseg + s];
            if (p.bias) l += p.bias[e_begin + tid];
            st_tagged(p.logits + e_begin + tid, l, tag);
        }
        // ------------------------------------------------------ phase 2
        if (warp == 0) {
            float lg[NJ];
            ld_tagged_all<NJ>(p.logits, lane, 32, p.E, tag, lg, status, &s_abort);
            int sel_e;
            float sel_p;
            softmax_topk_regs<NJ>(lg, p.E, k, (c == 0) ? p.probs : nullptr, lane, s_tk, sel_e, sel_p);
            if (sel_e < 0 || sel_e >= p.E) sel_e = -1;  // only after a timed-out poll; never dereferenced
            float norm = warp_sum(lane < k ? sel_p : 0.f);
            float wv = p.norm_topk ? sel_p / norm : sel_p;
            if (lane < k) {
                s_idx[lane] = sel_e;
                s_w[lane] = wv;
                if (c == 0) {
                    p.idx[lane] = sel_e;
                    p.w[lane] = wv;
                }
            }
        } else if (warp & 3) {
            convert_x(true);
        }
    } else {
        if (tid < k) {
            int e = ld_cg_i32(p.idx_in + tid);
            if (e < 0 || e >= p.E) {
                if (c == 0) record_error(status, MOE_ERR_BAD_INDEX);
                e = -1;
            }
            s_idx[tid] = e;
            s_w[tid] = ld_cg_f32(p.w_in + tid);
        }
        convert_x(false);
    }
    __syncthreads();

    // ---------------------------------------------------------- phase 3
    const int d_begin = (int)((long)c * D / G), d_end = (int)((long)(c + 1) * D / G);
    const int nrows = d_end - d_begin;
    // bulk copies of this CTA's down rows and their scales
    auto issue_down = [&]() {
        unsigned bytes = 0;
        for (int r = 0; r < k; r++)
            if (s_idx[r] >= 0) bytes += nrows * (rowF + nbF * (int)sizeof(ST));
        mbar_arrive_expect_tx(&s_bar, bytes);
        const uint8_t* DQ = reinterpret_cast<const uint8_t*>(p.down_q);
        const ST* DS = reinterpret_cast<const ST*>(p.down_s);
        if (nrows > 0) {
            for (int r = 0; r < k; r++) {
                int e = s_idx[r];
                if (e < 0) continue;
                size_t row0 = (size_t)e * D + d_begin;
                bulk_g2s(s_dq + (size_t)r * p.rows * rowF, DQ + row0 * rowF, nrows * rowF, &s_bar);
                bulk_g2s(s_ds + (size_t)r * p.rows * nbF, DS + row0 * nbF, nrows * nbF * (int)sizeof(ST), &s_bar);
            }
        }
    };

    const uint8_t* GQ = reinterpret_cast<const uint8_t*>(p.gate_q);
    const uint8_t* UQ = reinterpret_cast<const uint8_t*>(p.up_q);
    const ST* GS = reinterpret_cast<const ST*>(p.gate_s);
    const ST* US = reinterpret_cast<const ST*>(p.up_s);
    const int nchunk = rowD / 16;
    const long total = (long)k * F;
    const int g_begin = (int)((long)c * total / G), g_end = (int)((long)(c + 1) * total / G);

    auto load_pair = [&](int g, RowPair<QB, ST>& rp) {
        int r = g / F, n = g - r * F;
        int e = g < g_end ? s_idx[r] : -1;
        bool ok = e >= 0;
        size_t row = (size_t)(ok ? e : 0) * F + n;
#pragma unroll
        for (int j = 0; j < kNCH; j++) {
            int ci = j * 32 + lane;
            if (ok && ci < nchunk) {
                rp.g[j] = ld_stream16(GQ + row * rowD + 16 * ci);
                rp.u[j] = ld_stream16(UQ + row * rowD + 16 * ci);
                int blk = QB == 8 ? (ci >> 1) : ci;
                rp.gs[j] = ldg_nc(GS + row * nb + blk);
                rp.us[j] = ldg_nc(US + row * nb + blk);
            } else {
                rp.g[j] = rp.u[j] = make_uint4(0, 0, 0, 0);
                rp.gs[j] = rp.us[j] = ST(0.f);
            }
        }
    };
    auto finish_pair = [&](int g, const RowPair<QB, ST>& rp) {
        float ga = 0.f, ua = 0.f;
#pragma unroll
        for (int j = 0; j < kNCH; j++) {
            int ci = j * 32 + lane;
            if (ci < nchunk) {
                int ig, iu;
                float xs;
                if constexpr (QB == 8) {
                    uint4 hi = *reinterpret_cast<const uint4*>(s_xhi + 16 * ci);
                    uint4 lo = *reinterpret_cast<const uint4*>(s_xlo + 16 * ci);
                    ig = dot_i8_chunk(rp.g[j], hi, lo);
                    iu = dot_i8_chunk(rp.u[j], hi, lo);
                    xs = s_xs[ci >> 1];
                } else {
                    const uint4* H = reinterpret_cast<const uint4*>(s_xhi + 32 * ci);
                    const uint4* Lo = reinterpret_cast<const uint4*>(s_xlo + 32 * ci);
                    uint4 h0 = H[0], h1 = H[1], l0 = Lo[0], l1 = Lo[1];
                    ig = dot_i4_chunk(rp.g[j], h0, h1, l0, l1);
                    iu = dot_i4_chunk(rp.u[j], h0, h1, l0, l1);
                    xs = s_xs[ci] * (1.0f / 16.0f);
                }
                ga = fmaf((float)ig, to_f32(rp.gs[j]) * xs, ga);
                ua = fmaf((float)iu, to_f32(rp.us[j]) * xs, ua);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {  // both reductions interleaved
            ga += __shfl_xor_sync(kFull, ga, o);
            ua += __shfl_xor_sync(kFull, ua, o);
        }
        if (lane == 0 && g < g_end) p.h[g] = silu_mul(ga, ua);
    };

    {
        RowPair<QB, ST> A, B;
        int g = g_begin + warp;
        load_pair(g, A);
        // the down rows are requested together with the first gate/up rows so
        // that they stream concurrently; issued by a thread that never runs the
        // release fence of the exchange below (a fence may wait for them)
        if (tid == 32) issue_down();
        while (g < g_end) {
            int g2 = g + kFWarps;
            load_pair(g2, B);
            finish_pair(g, A);
            if (g2 >= g_end) break;
            int g3 = g2 + kFWarps;
            load_pair(g3, A);
            finish_pair(g2, B);
            g = g3;
        }
    }

    // ---------------------------------------------------------- phase 4
    // wait for every CTA's activations (one counter per launch parity; the
    // other one is cleared for the next launch). Each warp owns one slot: it
    // keeps that slot's activations for its pieces in registers (read once
    // from L2) and dots them with the staged down rows of its share of rows.
    arrive_and_wait(&p.hdr->hcount[s_seq & 1], (unsigned)G, status, &s_abort);
    mbar_wait(&s_bar, 0, status);

    const int wps = kFWarps / k;  // warps per slot (k <= 16)
    const int slot = warp / wps, sub = warp - slot * wps;
    if (slot < k && s_idx[slot] >= 0) {
        // The slot's activations, 8-byte pieces of codes per lane: piece pc
        // covers EPP consecutive units. They are turned into 16-bit fixed
        // point (as x is) with one power-of-two scale per block of 32 units,
        // the block max taken over the lanes holding the block, so that each
        // piece is dotted with integer dp4a.
        constexpr int EPP = QB == 8 ? 8 : 16;   // codes per 8-byte piece
        constexpr int NPL = QB == 8 ? 4 : 2;    // pieces per lane (F <= 1024)
        constexpr int LPB = kBlk / EPP;         // lanes per block: 4 or 2
        constexpr int NW = EPP / 4;             // plane words per piece and plane
        const int npieces = (QB == 8 ? F : F / 2) / 8;
        uint32_t hp[NPL][NW], lp[NPL][NW];
        float hsc[NPL];
#pragma unroll
        for (int i = 0; i < NPL; i++) {
            const int pc = i * 32 + lane;
            float v[EPP];
#pragma unroll
            for (int q = 0; q < EPP; q += 4) {
                uint4 t = pc < npieces ? ld_cg16(p.h + (size_t)slot * F + pc * EPP + q) : make_uint4(0, 0, 0, 0);
                v[q] = __uint_as_float(t.x);
                v[q + 1] = __uint_as_float(t.y);
                v[q + 2] = __uint_as_float(t.z);
                v[q + 3] = __uint_as_float(t.w);
            }
            float m = 0.f;
#pragma unroll
            for (int q = 0; q < EPP; q++) m = fmaxf(m, fabsf(v[q]));
#pragma unroll
            for (int o = 1; o < LPB; o <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
            const Fx f = fx_of_blockmax(m);
            hsc[i] = QB == 8 ? f.scale : f.scale * (1.0f / 16.0f);
#pragma unroll
            for (int w = 0; w < NW; w++) {
                uint32_t hw = 0, lw = 0;
#pragma unroll
                for (int bq = 0; bq < 4; bq++) {
                    // int8: byte bq of word w is unit 4w + bq; int4: word w
                    // holds the even units of its 8-unit group (w even) or the
                    // odd ones (w odd), as dot_i4_word expects
                    const int q = QB == 8 ? 4 * w + bq : 8 * (w >> 1) + 2 * bq + (w & 1);
                    const int X = fx_code(v[q], f.mul);
                    hw |= (uint32_t)((X >> 8) & 0xff) << (8 * bq);
                    lw |= (uint32_t)(X & 0xff) << (8 * bq);
                }
                hp[i][w] = hw;
                lp[i][w] = lw;
            }
        }
        const uint8_t* dq0 = s_dq + (size_t)slot * p.rows * rowF;
        const ST* ds0 = s_ds + (size_t)slot * p.rows * nbF;
        for (int row0 = sub; row0 < nrows; row0 += wps * kRU) {
            float acc[kRU];
#pragma unroll
            for (int u = 0; u < kRU; u++) {
                const int row = row0 + u * wps;
                acc[u] = 0.f;
                if (row < nrows) {
#pragma unroll
                    for (int i = 0; i < NPL; i++) {
                        const int pc = i * 32 + lane;
                        if (pc < npieces) {
                            const uint2 wv = *reinterpret_cast<const uint2*>(dq0 + (size_t)row * rowF + 8 * pc);
                            const float sc = to_f32(ds0[row * nbF + (EPP * pc) / kBlk]);
                            int hd = 0, ld = 0;
                            if constexpr (QB == 8) {
                                hd = dp4a_ss(wv.x, hp[i][0], hd);
                                hd = dp4a_ss(wv.y, hp[i][1], hd);
                                ld = dp4a_su(wv.x, lp[i][0], ld);
                                ld = dp4a_su(wv.y, lp[i][1], ld);
                            } else {
                                dot_i4_word(wv.x, hp[i][0], hp[i][1], lp[i][0], lp[i][1], hd, ld);
                                dot_i4_word(wv.y, hp[i][2], hp[i][3], lp[i][2], lp[i][3], hd, ld);
                            }
                            acc[u] = fmaf(sc * hsc[i], (float)(hd * 256 + ld), acc[u]);
                        }
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int u = 0; u < kRU; u++) acc[u] += __shfl_xor_sync(kFull, acc[u], o);
            if (lane == 0) {
#pragma unroll
                for (int u = 0; u < kRU; u++) {
                    const int row = row0 + u * wps;
                    if (row < nrows) s_part[row * k + slot] = acc[u];
                }
            }
        }
    }
    __syncthreads();
    if (tid < nrows) {
        float y = 0.f;
        for (int r = 0; r < k; r++)
            if (s_idx[r] >= 0) y = fmaf(s_w[r], s_part[tid * k + r], y);
        const int d = d_begin + tid;
        p.y[d] = y;
        if (p.x_next) {
            if constexpr (sizeof(XT) == 2)
                reinterpret_cast<__nv_bfloat16*>(p.x_next)[d] = __float2bfloat16_rn(s_x[d] + y);
            else
                reinterpret_cast<float*>(p.x_next)[d] = s_x[d] + y;
        }
    }
    // every CTA read the sequence number before producing anything CTA 0
    // waited for, so CTA 0 may advance it for the next launch
    if (c == 0 && tid == 0) atomicAdd(&p.hdr->seq, 1u);
}

// ------------------------------------------------------------- host side

static int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
}

static int pow2ceil(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Grid and per-CTA shape for one layer; false if the fused kernel cannot run it.
bool fused_plan(int E, int D, int F, int k, int qbits, int s_bytes, int x_bytes, bool has_router,
                FusedParams* fp, size_t* smem, int* grid) {
    int G = std::min(sm_count(), D);
    if (G < 1 || k > 16 || k < 1) return false;
    const int rows = (D + G - 1) / G;
    const int rowD = qbits == 8 ? D : D / 2, rowF = qbits == 8 ? F : F / 2;
    if (rowD / 16 > 32 * kNCH) return false;
    if (rowF / 8 > 32 * (qbits == 8 ? 4 : 2)) return false;
    if (F % 4) return false;
    if (((F / kBlk) * s_bytes) % 16) return false;  // bulk copies of whole scale rows
    if (has_router) {
        int nexp = (E + G - 1) / G;
        int nseg = kFWarps / pow2ceil(nexp);
        if (nseg < 1 || D % nseg) return false;
        int seg = D / nseg;
        int epc = 16 / x_bytes;
        if (seg % epc || seg / epc > 32 * kNRC) return false;
        fp->router_nseg = nseg;
        if (E > 1024) return false;
    } else {
        fp->router_nseg = 1;
    }
    FusedLayout L = fused_layout(D, F, k, qbits, s_bytes, rows);
    if (L.total > 200 * 1024) return false;
    fp->rows = rows;
    *smem = L.total;
    *grid = G;
    return true;
}

template <int QB, typename ST, typename XT>
static cudaError_t launch_fused_t(const FusedParams& p, int grid, size_t smem, cudaStream_t s) {
    const dim3 g(grid), b(kFThreads);
    switch (topk_nj(p.E, p.k)) {
        case 1: return launch(fused_layer_kernel<QB, ST, XT, 1>, g, b, smem, s, true, p);
        case 2: return launch(fused_layer_kernel<QB, ST, XT, 2>, g, b, smem, s, true, p);
        case 4: return launch(fused_layer_kernel<QB, ST, XT, 4>, g, b, smem, s, true, p);
        case 8: return launch(fused_layer_kernel<QB, ST, XT, 8>, g, b, smem, s, true, p);
        case 16: return launch(fused_layer_kernel<QB, ST, XT, 16>, g, b, smem, s, true, p);
        default: return launch(fused_layer_kernel<QB, ST, XT, 32>, g, b, smem, s, true, p);
    }
}

cudaError_t launch_fused(const FusedParams& p, int qbits, bool s_f16, bool x_bf16, int grid, size_t smem,
                         cudaStream_t s) {
    if (qbits == 8) {
        if (s_f16) return x_bf16 ? launch_fused_t<8, __half, __nv_bfloat16>(p, grid, smem, s)
                                  : launch_fused_t<8, __half, float>(p, grid, smem, s);
        return x_bf16 ? launch_fused_t<8, float, __nv_bfloat16>(p, grid, smem, s)
                      : launch_fused_t<8, float, float>(p, grid, smem, s);
    }
    if (s_f16) return x_bf16 ? launch_fused_t<4, __half, __nv_bfloat16>(p, grid, smem, s)
                              : launch_fused_t<4, __half, float>(p, grid, smem, s);
    return x_bf16 ? launch_fused_t<4, float, __nv_bfloat16>(p, grid, smem, s)
                  : launch_fused_t<4, float, float>(p, grid, smem, s);
}

}  // namespace moe
