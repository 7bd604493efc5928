// One whole MoE layer for one token in ONE persistent launch (decode), or a
// stack of such layers, one after the other, in one launch.
//
// lilting.ch "observing the Qwen MoE router" (section "hooking the router"):
// router logits -> fp32 softmax -> top-k. Qiita "custom Metal gather_qmm"
// (sections 4 and 7): only the k routed experts' rows are read, gate and up
// share x, down takes each slot's own activation, and the slots are combined
// with the routing weights. gist.science "Which expert misses are worth waiting
// for?" (method section): with a residency mask, a missed expert is kept when
// it is the first choice or its weight is >= the threshold, and is otherwise
// replaced by the best resident expert.
//
// Grid = one CTA of 16 warps per SM, all resident; the CTAs exchange small
// vectors through L2, each value or completion flag tagged with the launch's
// sequence number, so readers poll the data itself and no counter is shared:
//   0  before waiting on the previous launch: a bulk copy brings this CTA's
//      rows of the router weights (1-7 experts) into shared memory
//   1  x -> shared memory; the CTA's logits -> workspace (tagged); x -> 16-bit
//      fixed-point planes for the integer dots
//   2  every CTA polls the E logits (one or two per thread), takes the fp32
//      softmax with two block reductions, and selects the top k: each warp
//      extracts the k largest of its 32 probabilities (largest first, lower id
//      on equal values) with warp max-reductions, and warp 0 extracts the k
//      largest of those candidates. A residency mask adds the substitution:
//      each warp also extracts its 2k-1 best resident experts, from which warp
//      0 takes the replacements in rank order
//   3  one thread starts bulk copies of this CTA's rows of the k down
//      matrices into shared memory while the 16 warps stream this CTA's share
//      of the k*F gate/up row pairs from HBM (two row pairs in flight per warp)
//      and write h = silu(g)*u to the workspace; the CTA then raises its
//      completion flag
//   4  after every CTA's flag, the CTA reads all k*F activations once and
//      turns them into 16-bit fixed point (one power-of-two scale per block of
//      32 units); each warp dots its share of the (row, slot) pairs against the
//      staged down rows (integer dp4a); the CTA combines the k slots in slot
//      order, y[d] = sum_r w[r] * o_r[d], and writes x_next = x + y
// In a stack, layer l+1 starts when every CTA has raised its flag for layer l
// (its y and x_next are written): in chained mode its token is x_next of layer
// l, otherwise its own input, read only after that wait either way. The next
// layer's router rows are copied in while the current layer streams.
// Without a router (moe_decode) phases 0-2 are replaced by reading idx/w.
#include <mutex>

#include "dots.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace moe {

constexpr int kFThreads = 512;
constexpr int kFWarps = 16;
constexpr int kNRC = 4;  // router 16-byte chunks per lane
constexpr int kNCH = 4;  // gate/up 16-byte chunks per lane
constexpr int kDP = 4;   // (row, slot) down dots reduced together

struct FusedLayout {
    size_t x, xhi, xlo, xs, hhi, hlo, hs, wr, dq, ds, part, cand, rcand, total;
};

__host__ __device__ inline size_t fl_align(size_t v, size_t a) { return (v + a - 1) / a * a; }

// experts handled per CTA by the router phase
__host__ __device__ inline int fused_nexp(int E, int G) { return (E + G - 1) / G; }

__host__ __device__ inline FusedLayout fused_layout(int E, int D, int F, int k, int qbits, int s_bytes,
                                                    int x_bytes, int rows, int G) {
    FusedLayout L;
    size_t o = 0;
    const size_t rowF = qbits == 8 ? F : F / 2;
    const int nvw = (E + 31) / 32;  // warps of 32 experts in the selection
    L.x = o;     o = fl_align(o + sizeof(float) * D, 16);
    L.xhi = o;   o = fl_align(o + D, 16);
    L.xlo = o;   o = fl_align(o + D, 16);
    L.xs = o;    o = fl_align(o + sizeof(float) * (D / kBlk), 16);
    L.hhi = o;   o = fl_align(o + (size_t)k * F, 16);
    L.hlo = o;   o = fl_align(o + (size_t)k * F, 16);
    L.hs = o;    o = fl_align(o + sizeof(float) * (size_t)k * (F / kBlk), 16);
    L.wr = o;    o = fl_align(o + (size_t)fused_nexp(E, G) * D * x_bytes, 16);
    L.dq = o;    o = fl_align(o + (size_t)k * rows * rowF, 16);
    L.ds = o;    o = fl_align(o + (size_t)k * rows * (F / kBlk) * s_bytes, 16);
    L.part = o;  o = fl_align(o + sizeof(float) * (size_t)k * rows, 16);
    L.cand = o;  o = fl_align(o + sizeof(uint2) * (size_t)nvw * k, 16);
    L.rcand = o; o = fl_align(o + sizeof(uint2) * (size_t)nvw * (2 * k - 1), 16);
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

// Called by a whole warp whose lane l holds expert `e` (consecutive ids in
// lane order) with order key `key` (fp32 bits of its probability + 1, 0 for
// no expert): writes the n largest keys, largest first and the lower id first
// among equal keys, as {key, id} to out[0..n); missing entries are {0, 0}.
__device__ __forceinline__ void extract_top(unsigned key, int n, uint2* out, int e, int lane) {
    for (int it = 0; it < n; it++) {
        const unsigned m = __reduce_max_sync(kFull, key);
        if (m == 0u) {
            for (int i = it + lane; i < n; i += 32) out[i] = make_uint2(0u, 0u);
            return;
        }
        const unsigned tied = __ballot_sync(kFull, key == m);
        if (lane == __ffs(tied) - 1) {
            out[it] = make_uint2(m, (unsigned)e);
            key = 0u;
        }
    }
}

// Called by one warp: removes and returns the largest {key, id} of list[0..n)
// (lower id on equal keys); key 0 if the list is exhausted.
__device__ __forceinline__ uint2 take_best(uint2* list, int n, int lane) {
    unsigned bk = 0u, be = 0xffffffffu;
    int bi = -1;
    for (int i = lane; i < n; i += 32) {
        const uint2 cd = list[i];
        if (cd.x != 0u && (cd.x > bk || (cd.x == bk && cd.y < be))) {
            bk = cd.x;
            be = cd.y;
            bi = i;
        }
    }
    const unsigned m = __reduce_max_sync(kFull, bk);
    const unsigned me = __reduce_min_sync(kFull, bk == m ? be : 0xffffffffu);
    if (m != 0u && bi >= 0 && bk == m && be == me) list[bi].x = 0u;
    __syncwarp();
    return make_uint2(m, me);
}

template <int QB, typename ST, typename XT, int NL>
__global__ void __launch_bounds__(kFThreads, 1) fused_layer_kernel(const __grid_constant__ FusedArgs<NL> a) {
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ float s_rpart[kFWarps];
    __shared__ float s_rmax[kFWarps];
    __shared__ float s_rsum[kFWarps];
    __shared__ int s_idx[32];  // experts read per slot (after substitution), -1 = none
    __shared__ float s_w[32];
    __shared__ unsigned s_seq;
    __shared__ long long s_lim;
    __shared__ __align__(8) uint64_t s_bar;   // down rows of the current layer
    __shared__ __align__(8) uint64_t s_rbar;  // router rows of the next layer

    const FusedCommon& P = a.c;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int E = P.E, D = P.D, F = P.F, k = P.k;
    const int nb = D / kBlk, nbF = F / kBlk;
    const int rowD = QB == 8 ? D : D / 2;  // bytes of a gate/up row
    const int rowF = QB == 8 ? F : F / 2;  // bytes of a down row
    const FusedLayout Lo = fused_layout(E, D, F, k, QB, sizeof(ST), sizeof(XT), P.rows, G);
    float* s_x = reinterpret_cast<float*>(sm + Lo.x);
    int8_t* s_xhi = reinterpret_cast<int8_t*>(sm + Lo.xhi);
    uint8_t* s_xlo = sm + Lo.xlo;
    float* s_xs = reinterpret_cast<float*>(sm + Lo.xs);
    int8_t* s_hhi = reinterpret_cast<int8_t*>(sm + Lo.hhi);
    uint8_t* s_hlo = sm + Lo.hlo;
    float* s_hs = reinterpret_cast<float*>(sm + Lo.hs);
    const XT* s_wr = reinterpret_cast<const XT*>(sm + Lo.wr);
    uint8_t* s_dq = sm + Lo.dq;
    ST* s_ds = reinterpret_cast<ST*>(sm + Lo.ds);
    float* s_part = reinterpret_cast<float*>(sm + Lo.part);
    uint2* s_cand = reinterpret_cast<uint2*>(sm + Lo.cand);
    uint2* s_rcand = reinterpret_cast<uint2*>(sm + Lo.rcand);
    int* status = &P.hdr->status;
    unsigned* flag_h = P.flags;                  // activations of a layer written
    unsigned* flag_x = P.flags + kFusedMaxGrid;  // y / x_next of a layer written

    // this CTA's share: output rows (whole pairs), gate/up units, router experts
    const int d_begin = 2 * (int)((long)c * (D / 2) / G), d_end = 2 * (int)((long)(c + 1) * (D / 2) / G);
    const int nrows = d_end - d_begin;
    const long total = (long)k * F;
    const int g_begin = (int)((long)c * total / G), g_end = (int)((long)(c + 1) * total / G);
    const int e_begin = (int)((long)c * E / G), e_end = (int)((long)(c + 1) * E / G);
    const int nseg = P.router_nseg;
    const int rj = warp / nseg, rs = warp - rj * nseg;
    const int seg = D / nseg;
    const bool rvalid = P.has_router && e_begin + rj < e_end;
    constexpr int EPC = 16 / sizeof(XT);
    const int nvw = (E + 31) / 32;

    // bulk copy of this CTA's router rows (contiguous) of layer l
    auto request_router = [&](int l) {
        const unsigned bytes = (unsigned)((e_end - e_begin) * D * (int)sizeof(XT));
        mbar_arrive_expect_tx(&s_rbar, bytes);
        if (bytes) bulk_g2s(sm + Lo.wr, static_cast<const XT*>(a.L[l].W) + (size_t)e_begin * D, bytes, &s_rbar);
    };

    // ---------------------------------------------------------- phase 0
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        mbar_init(&s_rbar, 1);
        fence_barrier_init();
        if (P.has_router) request_router(0);
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    // the previous launch on this workspace has completed: its sequence
    // number increment is visible
    if (tid == 0) {
        s_seq = *reinterpret_cast<volatile unsigned*>(&P.hdr->seq);
        const unsigned long long lim = *reinterpret_cast<volatile unsigned long long*>(&P.hdr->wait_limit);
        s_lim = lim ? (long long)lim : kSpinLimitCycles;
    }
    __syncthreads();
    const unsigned seq0 = s_seq;
    const long long lim = s_lim;
    int router_next = P.has_router ? 0 : -1;  // layer whose router copy is requested and not waited for
    // this thread saw a wait run out; decisions on it are taken with
    // __syncthreads_or so that every thread of the CTA takes the same branch
    bool ab = false;

    for (int l = 0; l < P.nlayers; l++) {
        const FusedLayer& Y = a.L[l];
        const unsigned tag = seq_tag(seq0 + (unsigned)l);

        // ------------------------------------------------------ phase 1
        if (l > 0) {
            // every CTA has written layer l-1's y and x_next
            if (warp == 0 && !poll_flags(flag_x, G, seq_tag(seq0 + (unsigned)l - 1u), lim, status)) ab = true;
            if (__syncthreads_or(ab)) break;
        }
        const XT* X = reinterpret_cast<const XT*>((l > 0 && P.chain) ? a.L[l - 1].x_next : Y.x);
        for (int i = tid; i < D; i += kFThreads) s_x[i] = ldcg_f32(X + i);
        // residency of the experts this thread selects among
        const int e0 = tid, e1 = tid + kFThreads;
        const bool res0 = Y.resident && e0 < E && Y.resident[e0];
        const bool res1 = Y.resident && e1 < E && Y.resident[e1];
        __syncthreads();

        if (P.has_router) {
            if (!mbar_wait(&s_rbar, l & 1, status, lim)) {
                ab = true;
                mbar_wait(&s_rbar, l & 1, status);  // the copy must land before anything else happens
            }
            router_next = -1;
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kNRC; i++) {
                const int ci = i * 32 + lane;
                if (rvalid && ci * EPC < seg) {
                    const float* xs = s_x + rs * seg + ci * EPC;
                    const uint4 wq4 = *reinterpret_cast<const uint4*>(s_wr + (size_t)rj * D + rs * seg + ci * EPC);
                    const uint32_t* wq = reinterpret_cast<const uint32_t*>(&wq4);
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
                float lg = 0.f;
                for (int s2 = 0; s2 < nseg; s2++) lg += s_rpart[tid * nseg + s2];
                if (Y.bias) lg += Y.bias[e_begin + tid];
                st_tagged(P.logits + e_begin + tid, lg, tag);
            }
            // the next layer's router rows stream in while this layer runs
            if (tid == 0 && l + 1 < P.nlayers) request_router(l + 1);
            if (l + 1 < P.nlayers) router_next = l + 1;
        } else if (tid < k) {
            int e = ld_cg_i32(Y.idx_in + tid);
            if (e < 0 || e >= E) {
                if (c == 0) record_error(status, MOE_ERR_BAD_INDEX);
                e = -1;
            }
            s_idx[tid] = e;
            s_w[tid] = ld_cg_f32(Y.w_in + tid);
        }

        // x -> fixed-point planes (while the other CTAs' logits arrive)
        for (int b0 = warp; b0 < nb; b0 += kFWarps * 4) {
            float v[4];
            int blk[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                blk[i] = b0 + kFWarps * i;
                v[i] = blk[i] < nb ? s_x[blk[i] * kBlk + lane] : 0.f;
            }
            fx_store_blocks<4>(v, blk, nb, lane, QB, s_xhi, s_xlo, s_xs);
        }

        // ------------------------------------------------------ phase 2
        if (P.has_router) {
            float lg0 = -INFINITY, lg1 = -INFINITY;
            {
                bool r0 = e0 >= E, r1 = e1 >= E;
                const long long t0 = clock64();
                while (!(r0 && r1)) {
                    const uint64_t w0 = r0 ? 0ull : ld_tagged(P.logits + e0);
                    const uint64_t w1 = r1 ? 0ull : ld_tagged(P.logits + e1);
                    if (!r0 && tag_ok(w0, tag)) { r0 = true; lg0 = tag_val(w0); }
                    if (!r1 && tag_ok(w1, tag)) { r1 = true; lg1 = tag_val(w1); }
                    if (r0 && r1) break;
                    if (clock64() - t0 > lim) {
                        record_error(status, MOE_ERR_DEVICE_TIMEOUT);
                        ab = true;
                        break;
                    }
                }
            }
            // softmax: block max, then block sum of exp(l - max) in a fixed order
            float mx = warp_max(fmaxf(lg0, lg1));
            if (lane == 0) s_rmax[warp] = mx;
            __syncthreads();
            mx = s_rmax[0];
            for (int i = 1; i < kFWarps; i++) mx = fmaxf(mx, s_rmax[i]);
            float p0 = e0 < E ? expf(lg0 - mx) : 0.f;
            float p1 = e1 < E ? expf(lg1 - mx) : 0.f;
            const float ws = warp_sum(p0 + p1);
            if (lane == 0) s_rsum[warp] = ws;
            __syncthreads();
            float sum = 0.f;
            for (int i = 0; i < kFWarps; i++) sum += s_rsum[i];
            const float inv_s = 1.0f / sum;
            p0 *= inv_s;
            p1 *= inv_s;
            if (c == 0 && Y.probs) {
                if (e0 < E) Y.probs[e0] = p0;
                if (e1 < E) Y.probs[e1] = p1;
            }
            // per-warp candidates: the k largest of each warp's 32 experts (and
            // the 2k-1 largest resident ones)
#pragma unroll
            for (int j = 0; j < 2; j++) {
                const int vw = j * kFWarps + warp;
                if (vw < nvw) {
                    const int e = vw * 32 + lane;
                    const float pe = j ? p1 : p0;
                    const unsigned key = e < E ? __float_as_uint(pe) + 1u : 0u;
                    extract_top(key, k, s_cand + (size_t)vw * k, e, lane);
                    if (Y.resident) {
                        const bool re = j ? res1 : res0;
                        extract_top(re ? key : 0u, 2 * k - 1, s_rcand + (size_t)vw * (2 * k - 1), e, lane);
                    }
                }
            }
            __syncthreads();
            if (warp == 0) {
                int sel_e = -1;
                float sel_p = 0.f;
                for (int r = 0; r < k; r++) {
                    const uint2 b = take_best(s_cand, nvw * k, lane);
                    if (lane == r && b.x != 0u) {
                        sel_e = (int)b.y;
                        sel_p = __uint_as_float(b.x - 1u);
                    }
                }
                const float norm = warp_sum(lane < k ? sel_p : 0.f);
                const float wv = P.norm_topk ? sel_p / norm : sel_p;
                int use_e = sel_e;
                unsigned flg = 0;
                if (Y.resident) {
                    // replacement candidates: resident experts outside the chosen k
                    if (lane < k) s_idx[lane] = sel_e;
                    __syncwarp();
                    const int nrc = nvw * (2 * k - 1);
                    for (int i = lane; i < nrc; i += 32)
                        for (int r = 0; r < k; r++)
                            if (s_rcand[i].x != 0u && (int)s_rcand[i].y == s_idx[r]) s_rcand[i].x = 0u;
                    __syncwarp();
                    const bool my_res = lane < k && sel_e >= 0 && Y.resident[sel_e];
                    float mass = 0.f;
                    for (int r = 0; r < k; r++) {
                        const int er = __shfl_sync(kFull, sel_e, r);
                        const float wr = __shfl_sync(kFull, wv, r);
                        const bool rr = __shfl_sync(kFull, my_res, r);
                        int out = er;
                        unsigned f;
                        if (er < 0) {
                            f = 1;
                        } else if (rr) {
                            f = 0;
                        } else if (r == 0 || wr >= P.threshold) {
                            f = 1;
                        } else {
                            const uint2 b = take_best(s_rcand, nrc, lane);
                            if (b.x == 0u) {
                                f = 3;
                            } else {
                                out = (int)b.y;
                                f = 2;
                                mass += wr;
                            }
                        }
                        if (lane == r) {
                            use_e = out;
                            flg = f;
                        }
                    }
                    if (c == 0 && lane == 0 && Y.sub_mass) Y.sub_mass[0] = mass;
                }
                __syncwarp();
                if (lane < k) {
                    s_idx[lane] = use_e;
                    s_w[lane] = wv;
                    if (c == 0) {
                        Y.idx[lane] = sel_e;
                        Y.w[lane] = wv;
                        if (Y.idx_used) Y.idx_used[lane] = use_e;
                        if (Y.sub_flag) Y.sub_flag[lane] = (uint8_t)flg;
                    }
                }
            }
        }
        __syncthreads();

        // ------------------------------------------------------ phase 3
        // bulk copies of this CTA's down rows and their scales
        auto issue_down = [&]() {
            unsigned bytes = 0;
            for (int r = 0; r < k; r++)
                if (s_idx[r] >= 0) bytes += nrows * (rowF + nbF * (int)sizeof(ST));
            mbar_arrive_expect_tx(&s_bar, bytes);
            const uint8_t* DQ = reinterpret_cast<const uint8_t*>(Y.down_q);
            const ST* DS = reinterpret_cast<const ST*>(Y.down_s);
            if (nrows > 0) {
                for (int r = 0; r < k; r++) {
                    const int e = s_idx[r];
                    if (e < 0) continue;
                    const size_t row0 = (size_t)e * D + d_begin;
                    bulk_g2s(s_dq + (size_t)r * P.rows * rowF, DQ + row0 * rowF, nrows * rowF, &s_bar);
                    bulk_g2s(s_ds + (size_t)r * P.rows * nbF, DS + row0 * nbF, nrows * nbF * (int)sizeof(ST),
                             &s_bar);
                }
            }
        };

        const uint8_t* GQ = reinterpret_cast<const uint8_t*>(Y.gate_q);
        const uint8_t* UQ = reinterpret_cast<const uint8_t*>(Y.up_q);
        const ST* GS = reinterpret_cast<const ST*>(Y.gate_s);
        const ST* US = reinterpret_cast<const ST*>(Y.up_s);
        const int nchunk = rowD / 16;

        auto load_pair = [&](int g, RowPair<QB, ST>& rp) {
            const int r = g / F, n = g - r * F;
            const int e = g < g_end ? s_idx[r] : -1;
            const bool ok = e >= 0;
            const size_t row = (size_t)(ok ? e : 0) * F + n;
#pragma unroll
            for (int j = 0; j < kNCH; j++) {
                const int ci = j * 32 + lane;
                if (ok && ci < nchunk) {
                    rp.g[j] = ld_stream16(GQ + row * rowD + 16 * ci);
                    rp.u[j] = ld_stream16(UQ + row * rowD + 16 * ci);
                    const int blk = QB == 8 ? (ci >> 1) : ci;
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
                const int ci = j * 32 + lane;
                if (ci < nchunk) {
                    int ig, iu;
                    float xs;
                    if constexpr (QB == 8) {
                        const uint4 hi = *reinterpret_cast<const uint4*>(s_xhi + 16 * ci);
                        const uint4 lo = *reinterpret_cast<const uint4*>(s_xlo + 16 * ci);
                        ig = dot_i8_chunk(rp.g[j], hi, lo);
                        iu = dot_i8_chunk(rp.u[j], hi, lo);
                        xs = s_xs[ci >> 1];
                    } else {
                        const uint4* H = reinterpret_cast<const uint4*>(s_xhi + 32 * ci);
                        const uint4* Lw = reinterpret_cast<const uint4*>(s_xlo + 32 * ci);
                        const uint4 h0 = H[0], h1 = H[1], l0 = Lw[0], l1 = Lw[1];
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
            if (lane == 0 && g < g_end) P.h[g] = silu_mul(ga, ua);
        };

        {
            RowPair<QB, ST> A, B;
            int g = g_begin + warp;
            load_pair(g, A);
            // the down rows are requested together with the first gate/up rows
            if (tid == 32) issue_down();
            while (g < g_end) {
                const int g2 = g + kFWarps;
                load_pair(g2, B);
                finish_pair(g, A);
                if (g2 >= g_end) break;
                const int g3 = g2 + kFWarps;
                load_pair(g3, A);
                finish_pair(g2, B);
                g = g3;
            }
        }
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            st_release_u32(flag_h + c, tag);
        }

        // ------------------------------------------------------ phase 4
        if (warp == 0 && !poll_flags(flag_h, G, tag, lim, status)) ab = true;
        __syncthreads();
        // every slot's activations -> 16-bit fixed-point planes, one power-of-two
        // scale per block of 32 units (8 lanes of 4 units each)
        {
            const int n4 = (k * F) / 4;
            for (int i0 = warp * 32; i0 < n4; i0 += kFThreads) {
                const int i = i0 + lane;
                const bool ok = i < n4;
                const uint4 t = ok ? ld_cg16(P.h + 4 * i) : make_uint4(0, 0, 0, 0);
                const float v[4] = {__uint_as_float(t.x), __uint_as_float(t.y), __uint_as_float(t.z),
                                    __uint_as_float(t.w)};
                float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
                m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
                m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
                m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
                if (ok) {
                    const Fx f = fx_of_blockmax(m);
                    const int u = 4 * i;
                    if constexpr (QB == 8) {
                        uint32_t hw = 0, lw = 0;
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const int Xq = fx_code(v[q], f.mul);
                            hw |= (uint32_t)((Xq >> 8) & 0xff) << (8 * q);
                            lw |= (uint32_t)(Xq & 0xff) << (8 * q);
                        }
                        *reinterpret_cast<uint32_t*>(s_hhi + u) = hw;
                        *reinterpret_cast<uint32_t*>(s_hlo + u) = lw;
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const int Xq = fx_code(v[q], f.mul);
                            const int pos = fx_pos(u + q, 4);
                            s_hhi[pos] = (int8_t)(Xq >> 8);
                            s_hlo[pos] = (uint8_t)(Xq & 0xff);
                        }
                    }
                    if ((lane & 7) == 0) s_hs[u / kBlk] = QB == 8 ? f.scale : f.scale * (1.0f / 16.0f);
                }
            }
        }
        if (!mbar_wait(&s_bar, l & 1, status, lim)) {
            ab = true;
            mbar_wait(&s_bar, l & 1, status);  // the copies into this CTA's memory must land first
        }
        __syncthreads();

        // down: (row, slot) pairs q = i*k + r spread over the warps, 8-byte
        // pieces of a row per lane (int8: 8 units, int4: 16 units)
        {
            constexpr int EPP = QB == 8 ? 8 : 16;
            const int npieces = rowF / 8;
            const int npairs = nrows * k;
            for (int q0 = warp; q0 < npairs; q0 += kFWarps * kDP) {
                float acc[kDP];
#pragma unroll
                for (int u = 0; u < kDP; u++) {
                    acc[u] = 0.f;
                    const int q = q0 + u * kFWarps;
                    if (q < npairs) {
                        const int i = q / k, r = q - (q / k) * k;
                        if (s_idx[r] >= 0) {
                            const uint8_t* dq = s_dq + ((size_t)r * P.rows + i) * rowF;
                            const ST* ds = s_ds + ((size_t)r * P.rows + i) * nbF;
                            const int8_t* hh = s_hhi + (size_t)r * F;
                            const uint8_t* hl = s_hlo + (size_t)r * F;
                            const float* hs = s_hs + (size_t)r * nbF;
                            for (int pc = lane; pc < npieces; pc += 32) {
                                const uint2 wv = *reinterpret_cast<const uint2*>(dq + 8 * pc);
                                const int blk = (EPP * pc) / kBlk;
                                int hd = 0, ld = 0;
                                if constexpr (QB == 8) {
                                    const uint2 hp = *reinterpret_cast<const uint2*>(hh + 8 * pc);
                                    const uint2 lp = *reinterpret_cast<const uint2*>(hl + 8 * pc);
                                    hd = dp4a_ss(wv.x, hp.x, hd);
                                    hd = dp4a_ss(wv.y, hp.y, hd);
                                    ld = dp4a_su(wv.x, lp.x, ld);
                                    ld = dp4a_su(wv.y, lp.y, ld);
                                } else {
                                    const uint4 hp = *reinterpret_cast<const uint4*>(hh + 16 * pc);
                                    const uint4 lp = *reinterpret_cast<const uint4*>(hl + 16 * pc);
                                    dot_i4_word(wv.x, hp.x, hp.y, lp.x, lp.y, hd, ld);
                                    dot_i4_word(wv.y, hp.z, hp.w, lp.z, lp.w, hd, ld);
                                }
                                acc[u] = fmaf(to_f32(ds[blk]) * hs[blk], (float)(hd * 256 + ld), acc[u]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int u = 0; u < kDP; u++) acc[u] += __shfl_xor_sync(kFull, acc[u], o);
                if (lane == 0) {
#pragma unroll
                    for (int u = 0; u < kDP; u++) {
                        const int q = q0 + u * kFWarps;
                        if (q < npairs) s_part[q] = acc[u];
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
            Y.y[d] = y;
            if (Y.x_next) {
                if constexpr (sizeof(XT) == 2)
                    reinterpret_cast<__nv_bfloat16*>(Y.x_next)[d] = __float2bfloat16_rn(s_x[d] + y);
                else
                    reinterpret_cast<float*>(Y.x_next)[d] = s_x[d] + y;
            }
        }
        if (l + 1 < P.nlayers) {
            const bool any_ab = __syncthreads_or(ab);
            if (tid == 0) {
                __threadfence();
                st_release_u32(flag_x + c, tag);
            }
            if (any_ab) break;
        }
    }
    // a router copy requested for a layer that did not run must land before
    // this CTA's shared memory is released
    if (router_next >= 0) mbar_wait(&s_rbar, router_next & 1, status);
    __syncthreads();
    // every CTA read the sequence number before producing anything CTA 0
    // waited for, so CTA 0 may advance it past this launch's tags
    if (c == 0 && tid == 0) atomicAdd(&P.hdr->seq, (unsigned)P.nlayers);
}

// ------------------------------------------------------------- host side

int device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n;
    }
    return cache[dev];
}

static int pow2ceil(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Grid and per-CTA shape for one layer; false if the fused kernel cannot run it.
bool fused_plan(int E, int D, int F, int k, int qbits, int s_bytes, int x_bytes, bool has_router,
                FusedCommon* fc, size_t* smem, int* grid) {
    const int G = std::min(std::min(device_sm_count(), D / 2), kFusedMaxGrid);
    if (G < 1 || k < 1 || k > 32 || E < k || E > 2 * kFThreads) return false;
    const int rows = 2 * ((D / 2 + G - 1) / G);
    const int rowD = qbits == 8 ? D : D / 2;
    if (rowD / 16 > 32 * kNCH) return false;
    if (F % kBlk || D % kBlk) return false;
    if (((F / kBlk) * s_bytes) % 16) return false;  // bulk copies of whole scale rows
    if (has_router) {
        const int nexp = fused_nexp(E, G);
        const int nseg = kFWarps / pow2ceil(nexp);
        if (nseg < 1 || D % nseg) return false;
        const int seg = D / nseg;
        const int epc = 16 / x_bytes;
        if (seg % epc || seg / epc > 32 * kNRC) return false;
        fc->router_nseg = nseg;
    } else {
        fc->router_nseg = 1;
    }
    const FusedLayout L = fused_layout(E, D, F, k, qbits, s_bytes, x_bytes, rows, G);
    if (L.total > 220 * 1024) return false;
    fc->E = E;
    fc->D = D;
    fc->F = F;
    fc->k = k;
    fc->rows = rows;
    fc->has_router = has_router ? 1 : 0;
    *smem = L.total;
    *grid = G;
    return true;
}

template <int QB, typename ST, typename XT>
static cudaError_t launch_fused_t(const FusedCommon& fc, const FusedLayer* layers, int grid, size_t smem,
                                  cudaStream_t s) {
    const dim3 g(grid), b(kFThreads);
    if (fc.nlayers <= 1) {
        FusedArgs<1> a;
        a.c = fc;
        a.c.nlayers = 1;
        a.L[0] = layers[0];
        return launch(fused_layer_kernel<QB, ST, XT, 1>, g, b, smem, s, true, a);
    }
    if (fc.nlayers > kStackMax) return cudaErrorInvalidValue;
    FusedArgs<kStackMax> a = {};
    a.c = fc;
    for (int l = 0; l < fc.nlayers; l++) a.L[l] = layers[l];
    return launch(fused_layer_kernel<QB, ST, XT, kStackMax>, g, b, smem, s, true, a);
}

cudaError_t launch_fused(const FusedCommon& fc, const FusedLayer* layers, int qbits, bool s_f16, bool x_bf16,
                         int grid, size_t smem, cudaStream_t s) {
    if (qbits == 8) {
        if (s_f16) return x_bf16 ? launch_fused_t<8, __half, __nv_bfloat16>(fc, layers, grid, smem, s)
                                  : launch_fused_t<8, __half, float>(fc, layers, grid, smem, s);
        return x_bf16 ? launch_fused_t<8, float, __nv_bfloat16>(fc, layers, grid, smem, s)
                      : launch_fused_t<8, float, float>(fc, layers, grid, smem, s);
    }
    if (s_f16) return x_bf16 ? launch_fused_t<4, __half, __nv_bfloat16>(fc, layers, grid, smem, s)
                              : launch_fused_t<4, __half, float>(fc, layers, grid, smem, s);
    return x_bf16 ? launch_fused_t<4, float, __nv_bfloat16>(fc, layers, grid, smem, s)
                  : launch_fused_t<4, float, float>(fc, layers, grid, smem, s);
}

}  // namespace moe
