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
// Grid = one CTA of 16 warps per SM, all resident. The CTAs exchange three
// small vectors through L2 -- the logits, the activations and (in a stack) a
// layer's output -- as 64-bit words that carry a tag derived from the launch's
// sequence number next to the value. A reader polls the words themselves until
// each carries the current tag: no counter, flag or memory fence is involved.
//   0  before waiting on the previous launch: a bulk copy brings this CTA's
//      rows of the router weights (1-7 experts) into shared memory
//   1  x -> shared memory (in a stack, after the first layer: each warp stages
//      its 512-byte chunks of the previous layer's tagged x_next); each warp
//      dots its chunks of x with this CTA's router rows, and one thread per
//      expert adds the warps' shares in warp order and publishes the logit
//      (tagged); x -> 16-bit fixed-point planes for the integer dots
//   2  every CTA polls the E logits (one or two per thread) and selects the
//      top k by logit (softmax keeps the order): each warp ranks its 32 logits
//      (largest first, lower id on equal values) and keeps its k best as
//      candidates, which are then ranked among themselves; the block max and
//      the fp32 softmax sum are formed alongside, and the weights
//      exp(l - max)/sum are computed after the streaming. A residency mask adds
//      the substitution: each warp also ranks its 2k-1 best resident experts,
//      from which warp 0 takes the replacements in rank order, before streaming
//   3  the 16 warps stream this CTA's share of the k*F gate/up row pairs from
//      HBM (all of a warp's pairs requested at once: two in registers, a third
//      by cp.async into shared memory) and publish h = silu(g)*u (tagged); a
//      warp that streams two pairs then starts bulk copies of this CTA's rows
//      of the k down matrices into shared memory
//   4  each warp takes a (slot, share of the CTA's rows) task; the warps of a
//      slot read that slot's tagged activations with 16-byte loads and turn
//      each chunk, once complete, into 16-bit fixed point (one power-of-two
//      scale per block of 32 units), then, synchronised among themselves only,
//      hold the slot's activations in registers and dot them with the staged
//      down rows (integer dp4a), so a slot whose activations arrive early is
//      not held up by the others; the CTA combines the k slots in slot order,
//      y[d] = sum_r w[r] * o_r[d], and writes x_next = x + y
// In a stack, layer l+1 starts when every word of layer l's x_next has
// arrived: in chained mode those words are its token; otherwise its own token,
// copied in with its router rows while layer l streams, stands in for them
// chunk by chunk, so that the work waits as in a chain.
// Without a router (moe_decode) phases 0-2 are replaced by reading idx/w.
#include <mutex>

#include "dots.cuh"
#include "kernels.h"
#include "sync.cuh"
#include "tc.cuh"

namespace moe {

constexpr int kFThreads = 512;
constexpr int kFWarps = 16;
constexpr int kNCH = 4;      // gate/up 16-byte chunks per lane
constexpr int kDP = 8;       // down rows per warp task pass (computed together)
constexpr int kNPL = 4;      // 8-byte down pieces per lane (F <= 1024 int8, 2048 int4)
constexpr int kChunk = 128;  // tagged words per unit of the activation gather (1 KB)
constexpr int kXChunk = 64;  // tagged words per staged chunk of x (512 B)

// Shared-memory plan of one CTA.
struct FusedLayout {
    size_t x, xin, xhi, xlo, xs, hhi, hlo, hs, wr, dq, ds, part, cand, rcand, sel, stage;
    size_t total;
};

__host__ __device__ inline size_t fl_align(size_t v, size_t a) { return (v + a - 1) / a * a; }

// experts handled per CTA by the router phase
__host__ __device__ inline int fused_nexp(int E, int G) { return (E + G - 1) / G; }

// The staging region receives the tagged activations and (in a stack) the
// previous layer's output.
__host__ __device__ inline FusedLayout fused_layout(int E, int D, int F, int k, int qbits, int s_bytes,
                                                    int x_bytes, int rows, int G) {
    FusedLayout L;
    size_t o = 0;
    const size_t rowF = qbits == 8 ? F : F / 2;
    const int nvw = (E + 31) / 32;  // warps of 32 experts in the selection
    L.x = o;     o = fl_align(o + sizeof(float) * D, 16);
    L.xin = o;   o = fl_align(o + (size_t)x_bytes * D, 16);
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
    L.sel = o;   o = fl_align(o + sizeof(uint2) * 64, 16);
    L.stage = fl_align(o, 128);
    o = L.stage + sizeof(uint64_t) * (size_t)(k * F > D ? k * F : D);
    L.total = fl_align(o, 16);
    return L;
}

template <int QB, typename ST>
struct RowPair {
    uint4 g[kNCH], u[kNCH];
    ST gs[kNCH], us[kNCH];  // widened where used, so no load is waited for early
};

// Four consecutive activations v (units u..u+3, a lane's share of a block of
// 32 held by 8 lanes) -> the 16-bit fixed-point planes, one power-of-two scale
// per block. Called by a whole warp (ok: this lane's units exist).
template <int QB>
__device__ __forceinline__ void h_quad_to_planes(const float (&v)[4], int u, bool ok, int lane, int8_t* hhi,
                                                 uint8_t* hlo, float* hs) {
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
    m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
    if (!ok) return;
    const Fx f = fx_of_blockmax(m);
    if constexpr (QB == 8) {
        uint32_t hw = 0, lw = 0;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int Xq = fx_code(v[q], f.mul);
            hw |= (uint32_t)((Xq >> 8) & 0xff) << (8 * q);
            lw |= (uint32_t)(Xq & 0xff) << (8 * q);
        }
        *reinterpret_cast<uint32_t*>(hhi + u) = hw;
        *reinterpret_cast<uint32_t*>(hlo + u) = lw;
    } else {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int Xq = fx_code(v[q], f.mul);
            hhi[fx_pos(u + q, 4)] = (int8_t)(Xq >> 8);
            hlo[fx_pos(u + q, 4)] = (uint8_t)(Xq & 0xff);
        }
    }
    if ((lane & 7) == 0) hs[u / kBlk] = QB == 8 ? f.scale : f.scale * (1.0f / 16.0f);
}

// Fixed-point conversion of one block of 32 values held one per lane.
__device__ __forceinline__ void fx_store_block1(float v, int blk, int lane, int qbits, int8_t* hi, uint8_t* lo,
                                                float* scale) {
    const float m = warp_max(fabsf(v));
    const Fx f = fx_of_blockmax(m);
    const int X = fx_code(v, f.mul);
    const int pos = blk * kBlk + fx_pos(lane, qbits);
    hi[pos] = (int8_t)(X >> 8);
    lo[pos] = (uint8_t)(X & 0xff);
    if (lane == 0) scale[blk] = f.scale;
}

// Barrier over the nthreads threads (whole warps) that call it with this id.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Max and sum of the 16 per-warp partials, in a fixed order.
__device__ __forceinline__ float block_max16(const float* v) {
    float m2[4];
#pragma unroll
    for (int q = 0; q < 4; q++) m2[q] = fmaxf(fmaxf(v[4 * q], v[4 * q + 1]), fmaxf(v[4 * q + 2], v[4 * q + 3]));
    return fmaxf(fmaxf(m2[0], m2[1]), fmaxf(m2[2], m2[3]));
}
__device__ __forceinline__ float block_sum16(const float* v) {
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < kFWarps; i++) sum += v[i];
    return sum;
}

// Routing key of a logit: its fp32 bits mapped to an unsigned integer of the
// same order (negative values complemented, the sign bit set on the others),
// so that a larger logit has a larger key; 0 is kept for "no expert".
// Softmax is monotonic, so ranking logits ranks the probabilities.
__device__ __forceinline__ unsigned logit_key(float v) {
    const unsigned b = __float_as_uint(v);
    const unsigned u = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return u ? u : 1u;
}
__device__ __forceinline__ float key_logit(unsigned u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Candidate order: {logit key, id} (key 0: no expert); a ranks before b when
// its logit is larger, or equal with a lower id.
__device__ __forceinline__ int cand_before(uint2 a, uint2 b) {
    return (a.x > b.x || (a.x == b.x && a.y < b.y)) ? 1 : 0;
}

// Called by the whole CTA: writes the candidates of list[0..n) whose rank
// (number of entries ordered before them) is below k to out[rank] (and their
// ids to ids[rank] when ids is given). Eight
// threads share a candidate, each comparing it with every eighth entry.
__device__ __forceinline__ void rank_candidates(const uint2* list, int n, int k, uint2* out, int* ids, int tid) {
    const int q = tid & 7;
#pragma unroll 1
    for (int base = 0; base < n; base += kFThreads / 8) {
        const int i = base + (tid >> 3);
        const uint2 me = i < n ? list[i] : make_uint2(0u, 0u);
        int part = 0;
        if (me.x != 0u) {
#pragma unroll 4
            for (int j = q; j < n; j += 8) part += cand_before(list[j], me);
        }
        part += __shfl_xor_sync(kFull, part, 1);
        part += __shfl_xor_sync(kFull, part, 2);
        part += __shfl_xor_sync(kFull, part, 4);
        if (me.x != 0u && q == 0 && part < k) {
            out[part] = me;
            if (ids) ids[part] = (int)me.y;
        }
    }
}

// Called by a whole warp: brings the n tagged words src[0..n) of the chunks
// c = warp, warp + 16, ... (kXChunk words each) into dst (same offsets) by bulk
// copies, re-copying any chunk that still holds a word without `tag`, until
// every word of the warp's chunks carries it. Bounded by `lim`; on timeout
// records MOE_ERR_DEVICE_TIMEOUT and returns false (the copies in flight have
// landed by then).
__device__ __noinline__ bool warp_stage_tagged(uint64_t* dst, const uint64_t* src, int n, unsigned tag, uint64_t* bar,
                                  unsigned& phase, long long lim, int* status) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = (n + kXChunk - 1) / kXChunk;
    int mine = 0;
    for (int c = warp; c < nch; c += kFWarps) mine++;
    unsigned pending = mine >= 32 ? 0xffffffffu : ((1u << mine) - 1u);
    const long long t0 = clock64();
    bool ok = true;
#pragma unroll 1
    while (pending) {
        if (lane == 0) {
            unsigned bytes = 0;
            for (int i = 0; i < mine; i++)
                if (pending >> i & 1u) bytes += 8u * (unsigned)min(kXChunk, n - (warp + kFWarps * i) * kXChunk);
            mbar_arrive_expect_tx(bar, bytes);
            for (int i = 0; i < mine; i++) {
                if (!(pending >> i & 1u)) continue;
                const int c = warp + kFWarps * i;
                bulk_g2s(dst + (size_t)c * kXChunk, src + (size_t)c * kXChunk,
                         8u * (unsigned)min(kXChunk, n - c * kXChunk), bar);
            }
        }
        // the lanes agree on the outcome: the loop and the return are warp-uniform
        if (!__all_sync(kFull, mbar_wait(bar, phase, status, lim))) {
            mbar_wait(bar, phase, status);  // the copies must land before the memory is reused
            ok = false;
        }
        phase ^= 1u;
        unsigned still = 0;
#pragma unroll 1
        for (int i = 0; i < mine; i++) {
            if (!(pending >> i & 1u)) continue;
            const int c = warp + kFWarps * i;
            bool good = true;
#pragma unroll
            for (int q = 0; q < kXChunk / 32; q++) {
                const int wi = c * kXChunk + q * 32 + lane;
                if (wi < n) good &= tag_ok(dst[wi], tag);
            }
            if (!__all_sync(kFull, good)) still |= 1u << i;
        }
        pending = still;
        const bool late = __shfl_sync(kFull, clock64() - t0 > lim, 0);
        if (!ok || (pending && late)) {
            if (lane == 0 && ok) record_error(status, MOE_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
    return ok;
}

// Layer shape known at compile time (0 = read from the parameters): the
// kernel is instantiated for the decode shapes it serves most, so that every
// loop bound and shared-memory offset is a constant there.
template <int E_, int K_, int D_, int F_>
struct FShape {
    static constexpr int E = E_, k = K_, D = D_, F = F_;
};
using FRuntime = FShape<0, 0, 0, 0>;

template <int QB, typename ST, typename XT, int NL, class SH>
__global__ void __launch_bounds__(kFThreads, 1) fused_layer_kernel(const __grid_constant__ FusedArgs<NL> a) {
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ FusedLayer s_ly[2];  // this layer's and the next layer's pointers
    __shared__ float s_rpart[kFWarps * kFWarps];  // router shares [expert of this CTA][warp]
    __shared__ float s_rmax[kFWarps];
    __shared__ float s_rsum[kFWarps];
    __shared__ int s_idx[32];  // experts read per slot (after substitution), -1 = none
    __shared__ float s_w[32];
    __shared__ unsigned s_seq;
    __shared__ long long s_lim;
    __shared__ __align__(8) uint64_t s_bar;              // down rows of the current layer
    __shared__ __align__(8) uint64_t s_rbar;             // router rows
    __shared__ __align__(8) uint64_t s_wbar[kFWarps];    // per-warp staging

    const FusedCommon& P = a.c;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int E = SH::E ? SH::E : P.E, D = SH::D ? SH::D : P.D;
    const int F = SH::F ? SH::F : P.F, k = SH::k ? SH::k : P.k;
    const int nb = D / kBlk, nbF = F / kBlk;
    const int rowD = QB == 8 ? D : D / 2;  // bytes of a gate/up row
    const int rowF = QB == 8 ? F : F / 2;  // bytes of a down row
    const FusedLayout Lo = fused_layout(E, D, F, k, QB, sizeof(ST), sizeof(XT), P.rows, G);
    float* s_x = reinterpret_cast<float*>(sm + Lo.x);
    const XT* s_xin = reinterpret_cast<const XT*>(sm + Lo.xin);
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
    uint2* s_sel = reinterpret_cast<uint2*>(sm + Lo.sel);
    uint64_t* s_stage = reinterpret_cast<uint64_t*>(sm + Lo.stage);
    int* status = &P.hdr->status;

    // this CTA's share: output rows (whole pairs), gate/up units, router experts
    const int d_begin = 2 * (int)((long)c * (D / 2) / G), d_end = 2 * (int)((long)(c + 1) * (D / 2) / G);
    const int nrows = d_end - d_begin;
    const long total = (long)k * F;
    const int g_begin = (int)((long)c * total / G), g_end = (int)((long)(c + 1) * total / G);
    const int e_begin = (int)((long)c * E / G), e_end = (int)((long)(c + 1) * E / G);
    const int nvw = (E + 31) / 32;
    const int nxw = sizeof(XT) == 2 ? D / 2 : D;  // tagged words of a layer's x_next

    // one layer's pointers, from the kernel parameters into s_ly[b]
    auto load_layer = [&](int l, int b) {
        constexpr int NWD = sizeof(FusedLayer) / 4;
        const int t = tid - (kFThreads - 64);  // the last two warps
        if (t >= 0 && t < NWD)
            reinterpret_cast<uint32_t*>(&s_ly[b])[t] = reinterpret_cast<const uint32_t*>(&a.L[l])[t];
    };
    // bulk copy of this CTA's router rows (contiguous) of layer l
    // (and, for a later layer of an unchained stack, the layer's own x)
    auto request_router = [&](const FusedLayer& Y, bool with_x) {
        const unsigned bytes = (unsigned)((e_end - e_begin) * D * (int)sizeof(XT));
        const unsigned xbytes = with_x ? (unsigned)(D * (int)sizeof(XT)) : 0u;
        mbar_arrive_expect_tx(&s_rbar, bytes + xbytes);
        if (bytes) bulk_g2s(sm + Lo.wr, static_cast<const XT*>(Y.W) + (size_t)e_begin * D, bytes, &s_rbar);
        if (xbytes) bulk_g2s(sm + Lo.xin, Y.x, xbytes, &s_rbar);
    };

    // ---------------------------------------------------------- phase 0
    load_layer(0, 0);
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        mbar_init(&s_rbar, 1);
        for (int i = 0; i < kFWarps; i++) mbar_init(&s_wbar[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0 && P.has_router) request_router(s_ly[0], false);  // x may still be being written
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
    unsigned wph = 0;                         // this warp's staging-barrier phase
    // this thread saw a wait run out; decisions on it are taken with
    // __syncthreads_or so that every thread of the CTA takes the same branch
    bool ab = false;

#pragma unroll 1
    for (int l = 0; l < P.nlayers; l++) {
        const FusedLayer& Y = s_ly[l & 1];
        const unsigned tag = seq_tag(seq0 + (unsigned)l);
        // requested now, used later: the residency of the experts this thread
        // selects among, and the bias of the expert whose logit it completes
        const int e0 = tid, e1 = tid + kFThreads;
        const bool res0 = Y.resident && e0 < E && Y.resident[e0];
        const bool res1 = Y.resident && e1 < E && Y.resident[e1];
        const float bias_w = (P.has_router && Y.bias && tid < e_end - e_begin) ? Y.bias[e_begin + tid] : 0.f;

        // Called by warp 0 once the k slots are ranked: each slot's weight is
        // its softmax probability exp(l - max) / sum (the block max and the
        // fixed-order sum of the per-warp partials), renormalised over the k
        // when norm_topk; with residency, the substitution rule then sets the
        // slots' experts. Writes the slots' weights (and experts) to shared
        // memory and, in CTA 0, the routing outputs.
        auto route_weights = [&](bool resident) {
            const float mx = block_max16(s_rmax);
            const float inv_s = 1.0f / block_sum16(s_rsum);
            const uint2 sel = lane < k ? s_sel[lane] : make_uint2(0u, 0u);
            const int sel_e = sel.x ? (int)sel.y : -1;
            const float sel_p = sel.x ? expf(key_logit(sel.x) - mx) * inv_s : 0.f;
            const float norm = warp_sum(lane < k ? sel_p : 0.f);
            const float wv = P.norm_topk ? sel_p / norm : sel_p;
            int use_e = sel_e;
            unsigned flg = 0;
            if (resident) {
                const bool my_res = lane < k && sel_e >= 0 && Y.resident[sel_e];
                float mass = 0.f;
                int nrep = 0;  // replacements used so far
#pragma unroll 1
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
                        const uint2 b2 = nrep < k ? s_sel[32 + nrep] : make_uint2(0u, 0u);
                        if (b2.x == 0u) {
                            f = 3;
                        } else {
                            out = (int)b2.y;
                            f = 2;
                            mass += wr;
                            nrep++;
                        }
                    }
                    if (lane == r) {
                        use_e = out;
                        flg = f;
                    }
                }
                if (c == 0 && lane == 0 && Y.sub_mass) Y.sub_mass[0] = mass;
            }
            if (lane < k) {
                if (resident) s_idx[lane] = use_e;
                s_w[lane] = wv;
                if (c == 0) {
                    Y.idx[lane] = sel_e;
                    Y.w[lane] = wv;
                    if (Y.idx_used) Y.idx_used[lane] = use_e;
                    if (Y.sub_flag) Y.sub_flag[lane] = (uint8_t)flg;
                }
            }
        };

        // ------------------------------------------------------ phase 1
        // the router dots: each warp forms its share over its chunks of x (the
        // chunks it staged, as soon as they are in); one thread per expert of
        // this CTA adds the shares in warp order after the barrier
        auto router_shares = [&]() {
            __syncwarp();
            const int nexp = e_end - e_begin;
#pragma unroll 1
            for (int j = 0; j < nexp; j++) {
                const XT* wrow = s_wr + (size_t)j * D;
                float acc = 0.f;
#pragma unroll 1
                for (int i = warp * kXChunk + lane; i < nxw; i += kFWarps * kXChunk)
#pragma unroll
                    for (int q = 0; q < kXChunk; q += 32) {
                        const int wi = i + q;
                        if (wi < nxw) {
                            if constexpr (sizeof(XT) == 2) {
                                const uint32_t w2 = *reinterpret_cast<const uint32_t*>(wrow + 2 * wi);
                                acc = fmaf(bf16lo(w2), s_x[2 * wi], acc);
                                acc = fmaf(bf16hi(w2), s_x[2 * wi + 1], acc);
                            } else {
                                acc = fmaf(wrow[wi], s_x[wi], acc);
                            }
                        }
                    }
                acc = warp_sum(acc);
                if (lane == 0) s_rpart[j * kFWarps + warp] = acc;
            }
        };
        if (l > 0) {
            // layer l-1's x_next, tagged word by word by the CTAs that wrote it,
            // staged into shared memory: this layer starts when all of it has
            // arrived. Chained, it is this layer's token; unchained, the
            // layer's own token (copied in during the last layer) stands in
            // for it chunk by chunk, so that the work waits as in a chain.
            const unsigned ptag = seq_tag(seq0 + (unsigned)l - 1u);
            if (!warp_stage_tagged(s_stage, P.xex, nxw, ptag, &s_wbar[warp], wph, lim, status)) ab = true;
            if (P.has_router) {
                // the router rows (and the unchained token) of this layer
                if (!mbar_wait(&s_rbar, l & 1, status, lim)) {
                    ab = true;
                    mbar_wait(&s_rbar, l & 1, status);
                }
                router_next = -1;
            }
#pragma unroll 1
            for (int i = warp * kXChunk + lane; i < nxw; i += kFWarps * kXChunk)
#pragma unroll
                for (int q = 0; q < kXChunk; q += 32) {
                    const int wi = i + q;
                    if (wi < nxw) {
                        const uint32_t v = (uint32_t)s_stage[wi];
                        if constexpr (sizeof(XT) == 2) {
                            s_x[2 * wi] = P.chain ? bf16lo(v) : to_f32(s_xin[2 * wi]);
                            s_x[2 * wi + 1] = P.chain ? bf16hi(v) : to_f32(s_xin[2 * wi + 1]);
                        } else {
                            s_x[wi] = P.chain ? __uint_as_float(v) : s_xin[wi];
                        }
                    }
                }
            if (P.has_router) router_shares();
            if (__syncthreads_or(ab)) break;
        }
        if (l == 0 || (!P.chain && !P.has_router)) {
            const XT* X = reinterpret_cast<const XT*>(Y.x);
#pragma unroll 4
            for (int i = tid; i < D; i += kFThreads) s_x[i] = ldcg_f32(X + i);
            __syncthreads();
            if (l == 0 && P.has_router) {
                if (!mbar_wait(&s_rbar, 0, status, lim)) {
                    ab = true;
                    mbar_wait(&s_rbar, 0, status);
                }
                router_next = -1;
                router_shares();
                __syncthreads();
            }
        }

        if (P.has_router) {
            if (tid < e_end - e_begin) {
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < kFWarps; w++) acc += s_rpart[tid * kFWarps + w];
                st_tagged(P.logits + e_begin + tid, Y.bias ? acc + bias_w : acc, tag);
            }
        } else if (tid < k) {
            int e = ld_cg_i32(Y.idx_in + tid);
            if (e < 0 || e >= E) {
                if (c == 0) record_error(status, MOE_ERR_BAD_INDEX);
                e = -1;
            }
            s_idx[tid] = e;
            s_w[tid] = ld_cg_f32(Y.w_in + tid);
        }
        // the next layer's pointers (its router rows are requested once they are in)
        if (l + 1 < P.nlayers) load_layer(l + 1, (l + 1) & 1);

        // x -> fixed-point planes (while the other CTAs' logits arrive)
#pragma unroll 1
        for (int b = warp; b < nb; b += kFWarps) fx_store_block1(s_x[b * kBlk + lane], b, lane, QB, s_xhi, s_xlo, s_xs);

        // ------------------------------------------------------ phase 2
        if (P.has_router) {
            float lg0 = -INFINITY, lg1 = -INFINITY;
            {
                bool r0 = e0 >= E, r1 = e1 >= E;
                const long long t0 = clock64();
#pragma unroll 1
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
            // per-warp candidates, ranked by logit (the softmax keeps the
            // order): every lane counts the lanes of its warp whose key is
            // larger, the lower lane (lower id) first on equal keys; ranks below
            // k are kept (and below 2k-1 among resident experts, for the
            // replacements). The block max is formed alongside.
            {
                const float wmx = warp_max(fmaxf(lg0, lg1));
                if (lane == 0) s_rmax[warp] = wmx;
            }
#pragma unroll 1
            for (int j = 0; j < 2; j++) {
                const int vw = j * kFWarps + warp;
                if (vw < nvw) {
                    const int e = vw * 32 + lane;
                    const unsigned key = e < E ? logit_key(j ? lg1 : lg0) : 0u;
                    const bool re = Y.resident && (j ? res1 : res0);
                    const unsigned rkey = re ? key : 0u;
                    int rank = 0, rrank = 0;
                    if (Y.resident) {
#pragma unroll 8
                        for (int o = 0; o < 32; o++) {
                            // every lane executes both shuffles
                            const unsigned ko = __shfl_sync(kFull, key, o);
                            const int ro = __shfl_sync(kFull, (int)re, o);
                            const bool before = ko > key || (ko == key && o < lane);
                            rank += before;
                            rrank += (ro != 0 && (ko > rkey || (ko == rkey && o < lane))) ? 1 : 0;
                        }
                    } else {
#pragma unroll 8
                        for (int o = 0; o < 32; o++) {
                            const unsigned ko = __shfl_sync(kFull, key, o);
                            rank += (ko > key || (ko == key && o < lane)) ? 1 : 0;
                        }
                    }
                    uint2* cw = s_cand + (size_t)vw * k;
                    const int nvalid = __popc(__ballot_sync(kFull, key != 0u));
                    if (key != 0u && rank < k) cw[rank] = make_uint2(key, (unsigned)e);
                    for (int i = nvalid + lane; i < k; i += 32) cw[i] = make_uint2(0u, 0u);
                    if (Y.resident) {
                        uint2* rw = s_rcand + (size_t)vw * (2 * k - 1);
                        const int nres = __popc(__ballot_sync(kFull, rkey != 0u));
                        if (rkey != 0u && rrank < 2 * k - 1) rw[rrank] = make_uint2(key, (unsigned)e);
                        for (int i = nres + lane; i < 2 * k - 1; i += 32) rw[i] = make_uint2(0u, 0u);
                    }
                }
            }
            __syncthreads();
            // the k best candidates (eight threads per candidate, each comparing
            // with every eighth entry; without residency their ids are the
            // slots' experts), and alongside the softmax partial sums of
            // exp(l - max) in a fixed order
            rank_candidates(s_cand, nvw * k, k, s_sel, Y.resident ? nullptr : s_idx, tid);
            const float mx = block_max16(s_rmax);
            const float p0 = e0 < E ? expf(lg0 - mx) : 0.f;
            const float p1 = e1 < E ? expf(lg1 - mx) : 0.f;
            {
                const float ws = warp_sum(p0 + p1);
                if (lane == 0) s_rsum[warp] = ws;
            }
            __syncthreads();
            if (c == 0 && Y.probs) {
                const float inv_s = 1.0f / block_sum16(s_rsum);
                if (e0 < E) Y.probs[e0] = p0 * inv_s;
                if (e1 < E) Y.probs[e1] = p1 * inv_s;
            }
            if (Y.resident) {
                // replacement candidates: resident experts outside the chosen k,
                // ranked the same way; the best ones go to the replaced slots in
                // rank order
                const int RC = nvw * (2 * k - 1);
                if (tid < k) s_sel[32 + tid] = make_uint2(0u, 0u);
#pragma unroll 1
                for (int i = tid; i < RC; i += kFThreads) {
                    const unsigned e = s_rcand[i].y;
#pragma unroll 1
                    for (int r = 0; r < k; r++)
                        if (s_rcand[i].x != 0u && s_sel[r].y == e) s_rcand[i].x = 0u;
                }
                __syncthreads();
                rank_candidates(s_rcand, RC, k, s_sel + 32, nullptr, tid);
                __syncthreads();
                // the weights decide the substitutions, which decide the slots'
                // experts: done here, before the streaming
                if (warp == 0) route_weights(true);
            }
        }
        // the slots' experts are set (by the ranking, the substitution or the
        // given ids) before anything reads them
        if (!P.has_router || Y.resident) __syncthreads();

        // ------------------------------------------------------ phase 3
        // the warps stream their share of the gate/up row pairs with 16-byte
        // loads, two pairs in flight per warp, and publish h = silu(g)*u
        // (tagged); then one thread starts bulk copies of this CTA's rows of the
        // k down matrices (and, in a stack, the next layer's router rows)
        auto issue_down = [&]() {
            unsigned bytes = 0;
#pragma unroll 1
            for (int r = 0; r < k; r++)
                if (s_idx[r] >= 0) bytes += nrows * (rowF + nbF * (int)sizeof(ST));
            mbar_arrive_expect_tx(&s_bar, bytes);
            const uint8_t* DQ = reinterpret_cast<const uint8_t*>(Y.down_q);
            const ST* DS = reinterpret_cast<const ST*>(Y.down_s);
#pragma unroll 1
            for (int r = 0; r < k; r++) {
                const int e = s_idx[r];
                if (e < 0 || nrows == 0) continue;
                const size_t row0 = (size_t)e * D + d_begin;
                bulk_g2s(s_dq + (size_t)r * P.rows * rowF, DQ + row0 * rowF, nrows * rowF, &s_bar);
                bulk_g2s(s_ds + (size_t)r * P.rows * nbF, DS + row0 * nbF, nrows * nbF * (int)sizeof(ST), &s_bar);
            }
            // the next layer's router rows (its pointers were loaded before the last barrier)
            if (l + 1 < P.nlayers && P.has_router) request_router(s_ly[(l + 1) & 1], !P.chain);
        };
        if (l + 1 < P.nlayers && P.has_router) router_next = l + 1;

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
            for (int q = 0; q < kNCH; q++) {
                const int ci = q * 32 + lane;
                if (ok && ci < nchunk) {
                    rp.g[q] = ld_stream16(GQ + row * rowD + 16 * ci);
                    rp.u[q] = ld_stream16(UQ + row * rowD + 16 * ci);
                    const int blk = QB == 8 ? (ci >> 1) : ci;
                    rp.gs[q] = ldg_nc(GS + row * nb + blk);
                    rp.us[q] = ldg_nc(US + row * nb + blk);
                } else {
                    rp.g[q] = rp.u[q] = make_uint4(0, 0, 0, 0);
                    rp.gs[q] = rp.us[q] = ST(0.f);
                }
            }
        };
        auto finish_pair = [&](int g, const RowPair<QB, ST>& rp) {
            float ga = 0.f, ua = 0.f;
#pragma unroll
            for (int q = 0; q < kNCH; q++) {
                const int ci = q * 32 + lane;
                if (ci < nchunk) {
                    int ig, iu;
                    float xs;
                    if constexpr (QB == 8) {
                        const uint4 hi = *reinterpret_cast<const uint4*>(s_xhi + 16 * ci);
                        const uint4 lo = *reinterpret_cast<const uint4*>(s_xlo + 16 * ci);
                        ig = dot_i8_chunk(rp.g[q], hi, lo);
                        iu = dot_i8_chunk(rp.u[q], hi, lo);
                        xs = s_xs[ci >> 1];
                    } else {
                        const uint4* H = reinterpret_cast<const uint4*>(s_xhi + 32 * ci);
                        const uint4* Lw = reinterpret_cast<const uint4*>(s_xlo + 32 * ci);
                        const uint4 h0 = H[0], h1 = H[1], l0 = Lw[0], l1 = Lw[1];
                        ig = dot_i4_chunk(rp.g[q], h0, h1, l0, l1);
                        iu = dot_i4_chunk(rp.u[q], h0, h1, l0, l1);
                        xs = s_xs[ci] * (1.0f / 16.0f);
                    }
                    ga = fmaf((float)ig, to_f32(rp.gs[q]) * xs, ga);
                    ua = fmaf((float)iu, to_f32(rp.us[q]) * xs, ua);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {  // both reductions interleaved
                ga += __shfl_xor_sync(kFull, ga, o);
                ua += __shfl_xor_sync(kFull, ua, o);
            }
            if (lane == 0 && g < g_end) st_tagged(P.h + g, silu_mul(ga, ua), tag);
        };
        {
            // a warp's pairs are g0 + 16j; the first two go to registers, the
            // third is copied into this warp's slot of the staging region (idle
            // until the activation exchange) by cp.async at once, so every
            // pair of the warp is requested before any has arrived; further
            // pairs refill the registers
            const int g0 = g_begin + warp;
            const int pair_bytes = 2 * rowD + 2 * nb * (int)sizeof(ST);
            const bool third = g0 + 2 * kFWarps < g_end && (nb * (int)sizeof(ST)) % 16 == 0 &&
                               (warp + 1) * pair_bytes <= (int)(sizeof(uint64_t) * (size_t)(k * F > D ? k * F : D));
            uint8_t* slot = reinterpret_cast<uint8_t*>(s_stage) + (size_t)warp * pair_bytes;
            RowPair<QB, ST> A, B;
            load_pair(g0, A);
            load_pair(g0 + kFWarps, B);
            if (third) {
                const int g = g0 + 2 * kFWarps, r = g / F, n = g - r * F;
                const int e = s_idx[r];
                const size_t row = (size_t)(e >= 0 ? e : 0) * F + n;
                const int sbytes = nb * (int)sizeof(ST);
#pragma unroll 1
                for (int ci = lane; ci < nchunk; ci += 32) {
                    cp_async16(slot + 16 * ci, GQ + row * rowD + 16 * ci);
                    cp_async16(slot + rowD + 16 * ci, UQ + row * rowD + 16 * ci);
                }
#pragma unroll 1
                for (int ci = lane; ci < sbytes / 16; ci += 32) {
                    cp_async16(slot + 2 * rowD + 16 * ci, reinterpret_cast<const uint8_t*>(GS + row * nb) + 16 * ci);
                    cp_async16(slot + 2 * rowD + sbytes + 16 * ci,
                               reinterpret_cast<const uint8_t*>(US + row * nb) + 16 * ci);
                }
                cp_async_commit();
            }
            finish_pair(g0, A);
            finish_pair(g0 + kFWarps, B);
            int g = g0 + 2 * kFWarps;
            if (third) {
                cp_async_wait<0>();
                __syncwarp();
                RowPair<QB, ST> S;
                const ST* gsc = reinterpret_cast<const ST*>(slot + 2 * rowD);
                const ST* usc = gsc + nb;
#pragma unroll
                for (int q = 0; q < kNCH; q++) {
                    const int ci = q * 32 + lane;
                    const bool ok = ci < nchunk;
                    S.g[q] = ok ? *reinterpret_cast<const uint4*>(slot + 16 * ci) : make_uint4(0, 0, 0, 0);
                    S.u[q] = ok ? *reinterpret_cast<const uint4*>(slot + rowD + 16 * ci) : make_uint4(0, 0, 0, 0);
                    const int blk = QB == 8 ? (ci >> 1) : ci;
                    S.gs[q] = ok ? gsc[blk] : ST(0.f);
                    S.us[q] = ok ? usc[blk] : ST(0.f);
                }
                if (s_idx[g / F] < 0) {  // an expert slot without an id: nothing was meant to be read
#pragma unroll
                    for (int q = 0; q < kNCH; q++) {
                        S.g[q] = S.u[q] = make_uint4(0, 0, 0, 0);
                    }
                }
                finish_pair(g, S);
                g += kFWarps;
            }
            // pairs beyond those: two in flight in registers
            if (g < g_end) {
                load_pair(g, A);
#pragma unroll 1
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
        }
        // the down rows are requested by one thread of a warp that streams
        // the fewest pairs, once that warp's pairs are in: the gate/up bytes,
        // which the activation exchange waits for, go first, and the down rows
        // stream in during that exchange
        if (tid == (kFWarps - 2) * 32) issue_down();
        // without residency the weights are needed only by the combine: the
        // last warp, which also streams the fewest pairs, computes them
        if (P.has_router && !Y.resident && warp == kFWarps - 1) route_weights(false);
        __syncthreads();  // the staging region is free again
        // ------------------------------------------------------ phase 4
        // every slot's activations, gathered from the tagged words and turned
        // into 16-bit fixed point, one power-of-two scale per block of 32 units
        // (4 units per lane, 8 lanes per block)
        // with k * (16 / k) = 16 down tasks and whole chunks per slot, the two
        // (or more) warps of a slot's down tasks gather that slot's chunks
        // themselves and start its down dot as soon as they have them
        const int nsplit = k >= kFWarps ? 1 : kFWarps / k;
        const int cpr = F / kChunk;  // chunks per slot
        const bool by_slot = k * nsplit == kFWarps && F % kChunk == 0 && cpr % nsplit == 0;
        {
            // a warp's chunks are c = warp, warp + 16, ... (or its slot's share);
            // four units per lane, read with 16-byte loads straight into
            // registers (the bulk-copy engine is left to the down rows), up to
            // four chunks in flight, each converted as soon as all of its words
            // carry the tag
            const int nw_ = k * F;
            const int nch = (nw_ + kChunk - 1) / kChunk;
            const int mine = by_slot ? cpr / nsplit : (warp < nch ? (nch - warp + kFWarps - 1) / kFWarps : 0);
            const int cbase = by_slot ? (warp / nsplit) * cpr + (warp % nsplit) * (cpr / nsplit) : warp;
            const int cstep = by_slot ? 1 : kFWarps;
            const long long t0 = clock64();
            bool gave_up = false;  // warp-uniform
#pragma unroll 1
            for (int i0 = 0; i0 < mine && !gave_up; i0 += 4) {
                unsigned pend = 0;
#pragma unroll
                for (int i = 0; i < 4; i++)
                    if (i0 + i < mine) pend |= 1u << i;
#pragma unroll 1
                while (pend) {
                    uint64_t w[4][4];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int u = (cbase + cstep * (i0 + i)) * kChunk + 4 * lane;
                        if ((pend >> i & 1u) && u < nw_) {
                            ld_tagged2(P.h + u, w[i][0], w[i][1]);
                            ld_tagged2(P.h + u + 2, w[i][2], w[i][3]);
                        } else {
                            w[i][0] = w[i][1] = w[i][2] = w[i][3] = (uint64_t)tag << 32;
                        }
                    }
                    unsigned still = 0;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        if (!(pend >> i & 1u)) continue;
                        const int u = (cbase + cstep * (i0 + i)) * kChunk + 4 * lane;
                        const bool good = tag_ok(w[i][0], tag) && tag_ok(w[i][1], tag) && tag_ok(w[i][2], tag) &&
                                          tag_ok(w[i][3], tag);
                        if (!__all_sync(kFull, good)) {
                            still |= 1u << i;
                            continue;
                        }
                        const float v[4] = {tag_val(w[i][0]), tag_val(w[i][1]), tag_val(w[i][2]), tag_val(w[i][3])};
                        h_quad_to_planes<QB>(v, u, u < nw_, lane, s_hhi, s_hlo, s_hs);
                    }
                    pend = still;
                    if (pend && __shfl_sync(kFull, clock64() - t0 > lim, 0)) {
                        if (lane == 0) record_error(status, MOE_ERR_DEVICE_TIMEOUT);
                        ab = true;
                        gave_up = true;
                        break;
                    }
                }
            }
        }
        if (!mbar_wait(&s_bar, l & 1, status, lim)) {
            ab = true;
            mbar_wait(&s_bar, l & 1, status);  // the copies into this CTA's memory must land first
        }
        if (by_slot) {
            // the slot's warps (barrier ids 1..k, k <= 8); a slot of one warp needs none
            if (nsplit > 1) named_bar_sync(1 + warp / nsplit, 32 * nsplit);
            else __syncwarp();
        } else {
            __syncthreads();
        }

        // down: task = (slot, share of the CTA's rows); the warp keeps the
        // slot's activation planes in registers and dots them with each row
        // (8-byte pieces per lane: int8 8 units, int4 16 units)
        {
            constexpr int EPP = QB == 8 ? 8 : 16;
            constexpr int NW = EPP / 4;  // plane words per piece and plane
            const int npieces = rowF / 8;
            const int ntask = k * nsplit;
#pragma unroll 1
            for (int task = warp; task < ntask; task += kFWarps) {
                const int r = task / nsplit, part = task - r * nsplit;
                const int i0 = nrows * part / nsplit, i1 = nrows * (part + 1) / nsplit;
                if (s_idx[r] < 0 || i0 >= i1) continue;
                uint32_t hp[kNPL][NW], lp[kNPL][NW];
                float hsc[kNPL];
#pragma unroll
                for (int j = 0; j < kNPL; j++) {
                    const int pc = j * 32 + lane;
                    hsc[j] = 0.f;
#pragma unroll
                    for (int q = 0; q < NW; q++) hp[j][q] = lp[j][q] = 0u;
                    if (pc < npieces) {
                        const size_t o = (size_t)r * F + EPP * pc;
                        if constexpr (QB == 8) {
                            const uint2 h2 = *reinterpret_cast<const uint2*>(s_hhi + o);
                            const uint2 l2 = *reinterpret_cast<const uint2*>(s_hlo + o);
                            hp[j][0] = h2.x;
                            hp[j][1] = h2.y;
                            lp[j][0] = l2.x;
                            lp[j][1] = l2.y;
                        } else {
                            const uint4 h4 = *reinterpret_cast<const uint4*>(s_hhi + o);
                            const uint4 l4 = *reinterpret_cast<const uint4*>(s_hlo + o);
                            hp[j][0] = h4.x;
                            hp[j][1] = h4.y;
                            hp[j][2] = h4.z;
                            hp[j][3] = h4.w;
                            lp[j][0] = l4.x;
                            lp[j][1] = l4.y;
                            lp[j][2] = l4.z;
                            lp[j][3] = l4.w;
                        }
                        hsc[j] = s_hs[(size_t)r * nbF + (EPP * pc) / kBlk];
                    }
                }
                const uint8_t* dq0 = s_dq + (size_t)r * P.rows * rowF;
                const ST* ds0 = s_ds + (size_t)r * P.rows * nbF;
#pragma unroll 1
                for (int row0 = i0; row0 < i1; row0 += kDP) {
                    float acc[kDP];
#pragma unroll
                    for (int u = 0; u < kDP; u++) {
                        const int row = min(row0 + u, i1 - 1);  // past the end: a duplicate row, not stored
                        acc[u] = 0.f;
#pragma unroll
                        for (int j = 0; j < kNPL; j++) {
                            const int pc = j * 32 + lane;
                            if (pc < npieces) {
                                const uint2 wv = *reinterpret_cast<const uint2*>(dq0 + (size_t)row * rowF + 8 * pc);
                                const float sc = to_f32(ds0[row * nbF + (EPP * pc) / kBlk]);
                                int hd = 0, ld = 0;
                                if constexpr (QB == 8) {
                                    hd = dp4a_ss(wv.x, hp[j][0], hd);
                                    hd = dp4a_ss(wv.y, hp[j][1], hd);
                                    ld = dp4a_su(wv.x, lp[j][0], ld);
                                    ld = dp4a_su(wv.y, lp[j][1], ld);
                                } else {
                                    dot_i4_word(wv.x, hp[j][0], hp[j][1], lp[j][0], lp[j][1], hd, ld);
                                    dot_i4_word(wv.y, hp[j][2], hp[j][3], lp[j][2], lp[j][3], hd, ld);
                                }
                                acc[u] = fmaf(sc * hsc[j], (float)(hd * 256 + ld), acc[u]);
                            }
                        }
                    }
                    // the eight sums across the warp, halving the values a lane
                    // holds at each of the first three steps: lane bits 4, 3, 2
                    // pick the row a lane ends with
                    static_assert(kDP == 8, "the reduction below is written for 8 rows");
                    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
                    float a4[4], a2[2];
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const float send = b4 ? acc[j] : acc[j + 4];
                        a4[j] = (b4 ? acc[j + 4] : acc[j]) + __shfl_xor_sync(kFull, send, 16);
                    }
#pragma unroll
                    for (int j = 0; j < 2; j++) {
                        const float send = b3 ? a4[j] : a4[j + 2];
                        a2[j] = (b3 ? a4[j + 2] : a4[j]) + __shfl_xor_sync(kFull, send, 8);
                    }
                    float a1 = (b2 ? a2[1] : a2[0]) + __shfl_xor_sync(kFull, b2 ? a2[0] : a2[1], 4);
                    a1 += __shfl_xor_sync(kFull, a1, 2);
                    a1 += __shfl_xor_sync(kFull, a1, 1);
                    const int ru = (b4 ? 4 : 0) + (b3 ? 2 : 0) + (b2 ? 1 : 0);
                    if ((lane & 3) == 0 && row0 + ru < i1) s_part[(row0 + ru) * k + r] = a1;
                }
            }
        }
        __syncthreads();
        // combine, two rows per thread (a CTA's rows come in pairs):
        // y[d] = sum_r w[r] * o_r[d] in slot order, x_next = x + y; in a stack
        // the x_next pair is also published as one tagged word
        if (2 * tid < nrows) {
            const int d = d_begin + 2 * tid;
            float y0 = 0.f, y1 = 0.f;
#pragma unroll 4
            for (int r = 0; r < k; r++) {
                if (s_idx[r] >= 0) {
                    y0 = fmaf(s_w[r], s_part[(2 * tid) * k + r], y0);
                    y1 = fmaf(s_w[r], s_part[(2 * tid + 1) * k + r], y1);
                }
            }
            *reinterpret_cast<float2*>(Y.y + d) = make_float2(y0, y1);
            const bool publish = l + 1 < P.nlayers;
            if constexpr (sizeof(XT) == 2) {
                const __nv_bfloat162 xn = __floats2bfloat162_rn(s_x[d] + y0, s_x[d + 1] + y1);
                if (Y.x_next) *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(Y.x_next) + d) = xn;
                if (publish) st_tagged_u32(P.xex + d / 2, *reinterpret_cast<const uint32_t*>(&xn), tag);
            } else {
                const float x0 = s_x[d] + y0, x1 = s_x[d + 1] + y1;
                if (Y.x_next) *reinterpret_cast<float2*>(static_cast<float*>(Y.x_next) + d) = make_float2(x0, x1);
                if (publish) {
                    st_tagged(P.xex + d, x0, tag);
                    st_tagged(P.xex + d + 1, x1, tag);
                }
            }
        }
        if (l + 1 < P.nlayers && __syncthreads_or(ab)) break;
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

// Grid and per-CTA shape for one layer; false if the fused kernel cannot run it.
bool fused_plan(int E, int D, int F, int k, int qbits, int s_bytes, int x_bytes, bool has_router,
                FusedCommon* fc, size_t* smem, int* grid) {
    const int G = std::min(std::min(device_sm_count(), D / 2), kFusedMaxGrid);
    if (G < 1 || k < 1 || k > 32 || E < k || E > 2 * kFThreads) return false;
    if (F % kBlk || D % kBlk || (long)k * F > 32 * kFWarps * kChunk) return false;
    const int rows = 2 * ((D / 2 + G - 1) / G);
    const int rowD = qbits == 8 ? D : D / 2;
    if (rowD / 16 > 32 * kNCH) return false;
    if ((qbits == 8 ? F : F / 2) / 8 > 32 * kNPL) return false;
    // bulk copies of whole scale rows of the down matrices
    if (((F / kBlk) * s_bytes) % 16) return false;
    // one warp per router expert of a CTA
    if (has_router && fused_nexp(E, G) > kFWarps) return false;
    fc->router_nseg = 1;
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

template <int QB, typename ST, typename XT, class SH>
static cudaError_t launch_fused_t(const FusedCommon& fc, const FusedLayer* layers, int grid, size_t smem,
                                  cudaStream_t s) {
    const dim3 g(grid), b(kFThreads);
    if (fc.nlayers <= 1) {
        FusedArgs<1> a;
        a.c = fc;
        a.c.nlayers = 1;
        a.L[0] = layers[0];
        return launch(fused_layer_kernel<QB, ST, XT, 1, SH>, g, b, smem, s, true, a);
    }
    if (fc.nlayers > kStackMax) return cudaErrorInvalidValue;
    FusedArgs<kStackMax> a = {};
    a.c = fc;
    for (int l = 0; l < fc.nlayers; l++) a.L[l] = layers[l];
    return launch(fused_layer_kernel<QB, ST, XT, kStackMax, SH>, g, b, smem, s, true, a);
}

// The shapes with a compile-time instantiation: 256 experts top-8, d_model
// 2048, d_ff 768 (int8, fp16 scales, bf16 x) and 512 experts top-10, d_model
// 2048, d_ff 512 (int4, fp16 scales, bf16 x); everything else runs the
// runtime-shape instantiation.
template <int QB, typename ST, typename XT>
static cudaError_t launch_fused_shape(const FusedCommon& fc, const FusedLayer* layers, int grid, size_t smem,
                                      cudaStream_t s) {
    if constexpr (QB == 8 && sizeof(ST) == 2 && sizeof(XT) == 2) {
        if (fc.E == 256 && fc.k == 8 && fc.D == 2048 && fc.F == 768)
            return launch_fused_t<QB, ST, XT, FShape<256, 8, 2048, 768>>(fc, layers, grid, smem, s);
    }
    if constexpr (QB == 4 && sizeof(ST) == 2 && sizeof(XT) == 2) {
        if (fc.E == 512 && fc.k == 10 && fc.D == 2048 && fc.F == 512)
            return launch_fused_t<QB, ST, XT, FShape<512, 10, 2048, 512>>(fc, layers, grid, smem, s);
    }
    return launch_fused_t<QB, ST, XT, FRuntime>(fc, layers, grid, smem, s);
}

cudaError_t launch_fused(const FusedCommon& fc, const FusedLayer* layers, int qbits, bool s_f16, bool x_bf16,
                         int grid, size_t smem, cudaStream_t s) {
    if (qbits == 8) {
        if (s_f16) return x_bf16 ? launch_fused_shape<8, __half, __nv_bfloat16>(fc, layers, grid, smem, s)
                                  : launch_fused_shape<8, __half, float>(fc, layers, grid, smem, s);
        return x_bf16 ? launch_fused_shape<8, float, __nv_bfloat16>(fc, layers, grid, smem, s)
                      : launch_fused_shape<8, float, float>(fc, layers, grid, smem, s);
    }
    if (s_f16) return x_bf16 ? launch_fused_shape<4, __half, __nv_bfloat16>(fc, layers, grid, smem, s)
                              : launch_fused_shape<4, __half, float>(fc, layers, grid, smem, s);
    return x_bf16 ? launch_fused_shape<4, float, __nv_bfloat16>(fc, layers, grid, smem, s)
                  : launch_fused_shape<4, float, float>(fc, layers, grid, smem, s);
}

}  // namespace moe
