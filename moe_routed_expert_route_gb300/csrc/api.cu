// C ABI entry points: argument checks, workspace layout, kernel launches.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "kernels.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxDecodeT = 256;
// Up to this many tokens, one single-token layer launch per token is faster
// than the grouped products, even though an expert shared by the tokens is then
// read once per token (E=256 top-8 D=2048 F=768 int8: 14.3 us per token against
// 57 us for 4 tokens and 73 us for 8 tokens in the grouped products).
constexpr int kFusedTokens = 7;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Workspace sections, in bytes from the start. 0 = section not used.
struct Layout {
    size_t logits = 0, xq_hi = 0, xq_lo = 0, xq_s = 0, grp_expert = 0, grp_off = 0, assign = 0, h = 0;
    size_t xex = 0;
    size_t total = 0;
};

Layout layout(int op, int T, int k, int E, int D, int F) {
    Layout L;
    size_t off = sizeof(WsHeader);
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + std::max<size_t>(bytes, 1));
        return o;
    };
    const bool route = op == MOE_OP_ROUTE || op == MOE_OP_LAYER;
    const bool experts = op == MOE_OP_DECODE || op == MOE_OP_LAYER;
    // logits and h are sized for 64-bit tagged values (single-token layer kernel)
    if (route) L.logits = take(sizeof(uint64_t) * (size_t)T * E);
    if (experts) {
        size_t ng = (size_t)std::min(T * k, E);
        L.xq_hi = take((size_t)T * D);
        L.xq_lo = take((size_t)T * D);
        L.xq_s = take(sizeof(float) * (size_t)T * (D / kBlk));
        L.grp_expert = take(sizeof(int32_t) * ng);
        L.grp_off = take(sizeof(int32_t) * (ng + 1));
        L.assign = take(sizeof(int32_t) * (size_t)T * k);
        L.h = take(sizeof(uint64_t) * (size_t)T * k * F);
    }
    // a layer's x_next as tagged words (stacked single-token layers)
    if (experts) L.xex = take(sizeof(uint64_t) * (size_t)D);
    L.total = off;
    return L;
}

// Prefill workspace sections.
struct PLayout {
    size_t logits, idx, w, xh, pexp, chunk_cnt, chunk_base, cnt, off, gend, tgroup, tm0, tn, nmt, perm_tok, inv, hp, yp;
    size_t total;
    int nchunk, max_mtiles;
};

PLayout prefill_layout(int T, int k, int E, int D, int F) {
    PLayout L = {};
    size_t o = sizeof(WsHeader);
    auto take = [&](size_t bytes) {
        size_t r = o;
        o = align_up(o + std::max<size_t>(bytes, 1));
        return r;
    };
    const size_t n = (size_t)T * k;
    L.nchunk = (int)((n + kPermChunk - 1) / kPermChunk);
    L.max_mtiles = (int)((n + 127) / 128) + E;
    L.logits = take(sizeof(float) * (size_t)T * E);
    L.idx = take(sizeof(int32_t) * n);
    L.w = take(sizeof(float) * n);
    L.xh = take(2 * n * D);  // x rows in grouped order (fp16)
    L.pexp = take(sizeof(int32_t) * n);  // their power-of-two scale exponents
    L.chunk_cnt = take(sizeof(int32_t) * (size_t)L.nchunk * E);
    L.chunk_base = take(sizeof(int32_t) * (size_t)L.nchunk * E);
    L.cnt = take(sizeof(int32_t) * E);
    L.off = take(sizeof(int32_t) * (E + 1));
    L.gend = take(sizeof(int32_t) * E);
    L.tgroup = take(sizeof(int32_t) * L.max_mtiles);
    L.tm0 = take(sizeof(int32_t) * L.max_mtiles);
    L.tn = take(sizeof(int32_t) * L.max_mtiles);
    L.nmt = take(sizeof(int));
    L.perm_tok = take(sizeof(int32_t) * n);
    L.inv = take(sizeof(int32_t) * n);
    L.hp = take(2 * n * F);
    L.yp = take(sizeof(float) * n * D);
    L.total = o;
    return L;
}

// Grouped GEMM tiling: K stages of 64, gate/up tiles of 64 outputs, down
// tiles of 128 outputs.
bool prefill_shape_ok(int E, int D, int F) {
    return D % 128 == 0 && F % 64 == 0 && D >= 128 && F >= 64 && E <= 1024 && D <= 8192;
}

bool al16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

moe_status_t check_router(const moe_router_t* r, moe_dtype_t x_dtype) {
    if (!r) return MOE_ERR_INVALID_ARG;
    if (r->E < 1 || r->E > kMaxE || r->k < 1 || r->k > kMaxK || r->k > r->E) return MOE_ERR_INVALID_ARG;
    if (r->D < kBlk || r->D % kBlk) return MOE_ERR_INVALID_ARG;
    if (r->w_dtype != MOE_F32 && r->w_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (!al16(r->W)) return MOE_ERR_INVALID_ARG;
    if (r->bias && ((uintptr_t)r->bias & 3u)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status_t check_experts(const moe_experts_t* x, moe_dtype_t x_dtype, int k) {
    if (!x) return MOE_ERR_INVALID_ARG;
    if (x->E < 1 || x->E > kMaxE || k < 1 || k > kMaxK || k > x->E) return MOE_ERR_INVALID_ARG;
    if (x->D < kBlk || x->D % kBlk || x->F < kBlk || x->F % kBlk) return MOE_ERR_INVALID_ARG;
    if (x->q != MOE_Q_INT8_SYM_B32 && x->q != MOE_Q_INT4_SYM_B32) return MOE_ERR_UNSUPPORTED;
    if (x->s_dtype != MOE_F32 && x->s_dtype != MOE_F16) return MOE_ERR_UNSUPPORTED;
    if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    const void* ptrs[6] = {x->gate_q, x->gate_s, x->up_q, x->up_s, x->down_q, x->down_s};
    for (const void* p : ptrs)
        if (!al16(p)) return MOE_ERR_INVALID_ARG;
    int qbits = x->q == MOE_Q_INT8_SYM_B32 ? 8 : 4;
    if (!experts_supported(1, x->E, x->D, x->F, k, qbits)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

RouterParams router_params(const moe_router_t* r, const void* x, int T, int32_t* idx, float* w,
                           float* probs, void* ws, const Layout& L) {
    RouterParams p = {};
    p.T = T;
    p.E = r->E;
    p.D = r->D;
    p.k = r->k;
    p.norm_topk = r->norm_topk ? 1 : 0;
    p.W = r->W;
    p.bias = r->bias;
    p.x = x;
    p.logits = at<float>(ws, L.logits);
    p.idx = idx;
    p.w = w;
    p.probs = probs;
    p.hdr = at<WsHeader>(ws, 0);
    return p;
}

ExpertParams expert_params(const moe_experts_t* X, const void* x, moe_dtype_t x_dtype, int T, int k,
                           const int32_t* idx, const float* w, float* y, void* x_next, void* ws,
                           const Layout& L) {
    ExpertParams p = {};
    p.T = T;
    p.E = X->E;
    p.D = X->D;
    p.F = X->F;
    p.k = k;
    p.qbits = X->q == MOE_Q_INT8_SYM_B32 ? 8 : 4;
    p.s_f16 = X->s_dtype == MOE_F16;
    p.gate_q = X->gate_q;
    p.gate_s = X->gate_s;
    p.up_q = X->up_q;
    p.up_s = X->up_s;
    p.down_q = X->down_q;
    p.down_s = X->down_s;
    p.idx = idx;
    p.w = w;
    p.x = x;
    p.x_bf16 = x_dtype == MOE_BF16;
    p.hdr = at<WsHeader>(ws, 0);
    p.xq_hi = at<int8_t>(ws, L.xq_hi);
    p.xq_lo = at<uint8_t>(ws, L.xq_lo);
    p.xq_s = at<float>(ws, L.xq_s);
    p.grp_expert = at<int32_t>(ws, L.grp_expert);
    p.grp_off = at<int32_t>(ws, L.grp_off);
    p.assign = at<int32_t>(ws, L.assign);
    p.h = at<float>(ws, L.h);
    p.y = y;
    p.x_next = x_next;
    p.max_groups = std::min(T * k, X->E);
    return p;
}

FusedCommon fused_common(void* ws, const Layout& L) {
    FusedCommon f = {};
    f.nlayers = 1;
    f.hdr = at<WsHeader>(ws, 0);
    f.logits = L.logits ? at<uint64_t>(ws, L.logits) : nullptr;
    f.h = at<uint64_t>(ws, L.h);
    f.xex = at<uint64_t>(ws, L.xex);
    return f;
}

FusedLayer fused_layer(const moe_experts_t* X, const void* x, float* y, void* x_next) {
    FusedLayer f = {};
    f.x = x;
    f.gate_q = X->gate_q;
    f.gate_s = X->gate_s;
    f.up_q = X->up_q;
    f.up_s = X->up_s;
    f.down_q = X->down_q;
    f.down_s = X->down_s;
    f.y = y;
    f.x_next = x_next;
    return f;
}

int qbits_of(const moe_experts_t* X) { return X->q == MOE_Q_INT8_SYM_B32 ? 8 : 4; }
int scale_bytes(const moe_experts_t* X) { return X->s_dtype == MOE_F16 ? 2 : 4; }

// Routing of many tokens: tensor-core logits + one warp per token when the
// shapes allow, else the CUDA-core router kernel.
moe_status_t route_many(const moe_router_t* router, const void* x, moe_dtype_t x_dtype, int T, int32_t* idx_buf,
                        float* w_buf, float* probs, float* logits, WsHeader* hdr, cudaStream_t s) {
    const int E = router->E, D = router->D, k = router->k;
    cudaError_t e;
    if (x_dtype == MOE_BF16 && router->w_dtype == MOE_BF16 && E % 128 == 0 && D % 64 == 0) {
        GemmParams g = {};
        if (!make_tmap_2d(&g.tmA, 2, x, D, T, 2ull * D, 64, 128, 128) ||
            !make_tmap_2d(&g.tmB0, 2, router->W, D, E, 2ull * D, 64, 128, 128))
            return MOE_ERR_CUDA;
        g.K = D;
        g.rows_per_ntile = 128;
        g.n_mtiles = (T + 127) / 128;
        g.m_total = T;
        g.n_ntiles = E / 128;
        g.C = logits;
        g.ldc = E;
        g.hdr = hdr;
        e = launch_router_gemm(g, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        TopkParams tp = {T, E, k, router->norm_topk ? 1 : 0, logits, router->bias, idx_buf, w_buf, probs};
        e = launch_topk(tp, s);
    } else {
        RouterParams rp = {};
        rp.T = T;
        rp.E = E;
        rp.D = D;
        rp.k = k;
        rp.norm_topk = router->norm_topk ? 1 : 0;
        rp.W = router->W;
        rp.bias = router->bias;
        rp.x = x;
        rp.logits = logits;
        rp.idx = idx_buf;
        rp.w = w_buf;
        rp.probs = probs;
        rp.hdr = hdr;
        e = launch_router(rp, router->w_dtype == MOE_BF16, x_dtype == MOE_BF16, s, true);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

// The routed experts of many tokens as grouped tensor-core products: stable
// grouping of the (token, slot) assignments by expert, x gathered in grouped
// order, gate/up with SwiGLU, down, and the weighted un-permute (y, and
// x_next = x + y when x_next is given).
moe_status_t grouped_experts(const moe_experts_t* experts, const void* x, moe_dtype_t x_dtype, int T, int k,
                             const int32_t* idx_buf, const float* w_buf, float* y, void* x_next, int32_t* counts,
                             int32_t* perm, void* workspace, const PLayout& P, cudaStream_t s) {
    const int E = experts->E, D = experts->D, F = experts->F;
    WsHeader* hdr = at<WsHeader>(workspace, 0);
    cudaError_t e;
    const int nt = kEgTile;  // token tile of the expert products
    PermParams pp = {};
    pp.tile_rows = nt;
    pp.n = T * k;
    pp.k = k;
    pp.E = E;
    pp.nchunk = P.nchunk;
    pp.idx = idx_buf;
    pp.hdr = hdr;
    pp.chunk_cnt = at<int32_t>(workspace, P.chunk_cnt);
    pp.chunk_base = at<int32_t>(workspace, P.chunk_base);
    pp.cnt = at<int32_t>(workspace, P.cnt);
    pp.off = at<int32_t>(workspace, P.off);
    pp.group_end = at<int32_t>(workspace, P.gend);
    pp.counts_out = counts;
    pp.tile_group = at<int32_t>(workspace, P.tgroup);
    pp.tile_m0 = at<int32_t>(workspace, P.tm0);
    pp.tile_n = at<int32_t>(workspace, P.tn);
    pp.n_mtiles = at<int>(workspace, P.nmt);
    pp.perm_tok = at<int32_t>(workspace, P.perm_tok);
    pp.perm_out = perm;
    pp.inv = at<int32_t>(workspace, P.inv);
    e = launch_perm(pp, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    const long n = (long)T * k;
    void* xp = at<void>(workspace, P.xh);
    void* hp = at<void>(workspace, P.hp);
    void* yp = at<void>(workspace, P.yp);
    int32_t* pexp = at<int32_t>(workspace, P.pexp);
    e = launch_gather_f16(x, x_dtype == MOE_BF16, pp.perm_tok, (int)n, D, xp, pexp, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    const int qbits = qbits_of(experts);
    const int cb = qbits == 8 ? 1 : 2;  // codes per byte
    const unsigned rb = 64 / cb;        // code bytes per row per K stage
    const bool sf16 = experts->s_dtype == MOE_F16;
    const int sms = device_sm_count();
    EgParams g1 = {};
    if (!make_tmap_2d(&g1.tmX, 1, xp, D, n, 2ull * D, 64, nt, 128) ||
        !make_tmap_2d(&g1.tmXh, 1, xp, D, n, 2ull * D, 64, nt / 2, 128) ||
        !make_tmap_2d(&g1.tmW0, 0, experts->gate_q, D / cb, (unsigned long long)E * F, D / cb, rb, 64, rb) ||
        !make_tmap_2d(&g1.tmW1, 0, experts->up_q, D / cb, (unsigned long long)E * F, D / cb, rb, 64, rb))
        return MOE_ERR_CUDA;
    g1.S0 = experts->gate_s;
    g1.S1 = experts->up_s;
    g1.K = D;
    g1.w_rows = F;
    g1.nwb = F / 64;
    g1.tile_group = pp.tile_group;
    g1.tile_m0 = pp.tile_m0;
    g1.tile_n = pp.tile_n;
    g1.n_tiles_dev = pp.n_mtiles;
    g1.C = hp;
    g1.ldc = F;
    g1.pexp = pexp;
    g1.hdr = hdr;
    e = launch_egemm(g1, qbits, sf16, true, sms, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    EgParams g2 = g1;
    if (!make_tmap_2d(&g2.tmX, 1, hp, F, n, 2ull * F, 64, nt, 128) ||
        !make_tmap_2d(&g2.tmXh, 1, hp, F, n, 2ull * F, 64, nt / 2, 128) ||
        !make_tmap_2d(&g2.tmW0, 0, experts->down_q, F / cb, (unsigned long long)E * D, F / cb, rb, 64, rb))
        return MOE_ERR_CUDA;
    g2.tmW1 = g2.tmW0;
    g2.S0 = experts->down_s;
    g2.S1 = experts->down_s;
    g2.K = F;
    g2.w_rows = D;
    g2.nwb = D / 128;
    g2.C = yp;
    g2.ldc = D;
    e = launch_egemm(g2, qbits, sf16, false, sms, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    CombineParams cp = {T, D, k, pp.inv, w_buf, static_cast<const float*>(yp), y, x, x_dtype == MOE_BF16 ? 1 : 0, x_next};
    return from_cuda(launch_combine(cp, s));
}

// Offset of the probabilities that substitution reads when the caller passes
// none (after every other section of a layer workspace).
size_t layer_bytes(int T, int k, int E, int D, int F) {
    size_t bytes = layout(MOE_OP_LAYER, T, k, E, D, F).total;
    // several tokens through the grouped products
    if (T >= 2 && prefill_shape_ok(E, D, F)) bytes = std::max(bytes, prefill_layout(T, k, E, D, F).total);
    return align_up(bytes);
}

// One layer for T tokens, with an optional residency substitution between the
// routing and the experts.
moe_status_t layer_impl(const moe_router_t* router, const moe_experts_t* experts, const void* x,
                        moe_dtype_t x_dtype, int T, const uint8_t* resident, float threshold, int32_t* idx,
                        float* w, float* probs, int32_t* idx_used, uint8_t* sub_flag, float* sub_mass, float* y,
                        void* x_next, void* workspace, size_t ws_bytes, cudaStream_t s) {
    moe_status_t st = check_router(router, x_dtype);
    if (st != MOE_OK) return st;
    st = check_experts(experts, x_dtype, router->k);
    if (st != MOE_OK) return st;
    if (router->E != experts->E || router->D != experts->D) return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > kMaxDecodeT || !al16(x) || !idx || !w || !al16(y)) return MOE_ERR_INVALID_ARG;
    if (x_next && !al16(x_next)) return MOE_ERR_INVALID_ARG;
    const int k = router->k, E = experts->E, D = experts->D, F = experts->F;
    Layout L = layout(MOE_OP_LAYER, T, k, E, D, F);
    if (!workspace || ((uintptr_t)workspace & (kAlign - 1)) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (T <= kFusedTokens && (router->w_dtype == MOE_BF16) == (x_dtype == MOE_BF16)) {
        FusedCommon fc = fused_common(workspace, L);
        size_t smem = 0;
        int grid = 0;
        if (fused_plan(E, D, F, k, qbits_of(experts), scale_bytes(experts), x_dtype == MOE_BF16 ? 2 : 4, true,
                       &fc, &smem, &grid)) {
            fc.norm_topk = router->norm_topk ? 1 : 0;
            fc.threshold = threshold;
            const size_t xb = x_dtype == MOE_BF16 ? 2 : 4;
            for (int t = 0; t < T; t++) {  // one single-token launch per token
                FusedLayer ly = fused_layer(experts, static_cast<const char*>(x) + (size_t)t * D * xb,
                                            y + (size_t)t * D,
                                            x_next ? static_cast<char*>(x_next) + (size_t)t * D * xb : nullptr);
                ly.W = router->W;
                ly.bias = router->bias;
                ly.idx = idx + (size_t)t * k;
                ly.w = w + (size_t)t * k;
                ly.probs = probs ? probs + (size_t)t * E : nullptr;
                if (resident) {
                    ly.resident = resident;
                    ly.idx_used = idx_used + (size_t)t * k;
                    ly.sub_flag = sub_flag + (size_t)t * k;
                    ly.sub_mass = sub_mass + t;
                }
                cudaError_t e = launch_fused(fc, &ly, qbits_of(experts), experts->s_dtype == MOE_F16,
                                             x_dtype == MOE_BF16, grid, smem, s);
                if (e != cudaSuccess) return MOE_ERR_CUDA;
            }
            return MOE_OK;
        }
    }
    float* sub_probs = probs;
    if (resident && !probs) {
        if (ws_bytes < layer_bytes(T, k, E, D, F) + sizeof(float) * (size_t)T * E) return MOE_ERR_WORKSPACE;
        sub_probs = at<float>(workspace, layer_bytes(T, k, E, D, F));
    }
    // the substituted routing (weights unchanged: a replacement keeps its slot's weight)
    auto substitute = [&]() {
        SubstituteParams sp = {T, E, k, sub_probs, idx, w, resident, threshold, idx_used, w, sub_flag, sub_mass};
        return launch_substitute(sp, s);
    };
    if (T >= 2 && prefill_shape_ok(E, D, F)) {
        PLayout P = prefill_layout(T, k, E, D, F);
        if (ws_bytes < P.total) return MOE_ERR_WORKSPACE;
        moe_status_t rs = route_many(router, x, x_dtype, T, idx, w, sub_probs, at<float>(workspace, P.logits),
                                     at<WsHeader>(workspace, 0), s);
        if (rs != MOE_OK) return rs;
        if (resident && substitute() != cudaSuccess) return MOE_ERR_CUDA;
        return grouped_experts(experts, x, x_dtype, T, k, resident ? idx_used : idx, w, y, x_next, nullptr,
                               nullptr, workspace, P, s);
    }
    RouterParams rp = router_params(router, x, T, idx, w, sub_probs, workspace, L);
    ExpertParams ep = expert_params(experts, x, x_dtype, T, k, resident ? idx_used : idx, w, y, x_next,
                                    workspace, L);
    if (!resident) {
        // the router's last CTA also builds the expert kernels' inputs
        rp.xq_hi = const_cast<int8_t*>(ep.xq_hi);
        rp.xq_lo = const_cast<uint8_t*>(ep.xq_lo);
        rp.xq_s = const_cast<float*>(ep.xq_s);
        rp.qbits = ep.qbits;
        rp.grp_expert = const_cast<int32_t*>(ep.grp_expert);
        rp.grp_off = const_cast<int32_t*>(ep.grp_off);
        rp.assign = const_cast<int32_t*>(ep.assign);
    }
    cudaError_t e = launch_router(rp, router->w_dtype == MOE_BF16, x_dtype == MOE_BF16, s, true);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (resident) {
        if (substitute() != cudaSuccess) return MOE_ERR_CUDA;
        PrepParams pp = {};
        pp.T = T;
        pp.E = E;
        pp.D = D;
        pp.k = k;
        pp.qbits = ep.qbits;
        pp.x = x;
        pp.x_bf16 = ep.x_bf16;
        pp.idx = idx_used;
        pp.hdr = ep.hdr;
        pp.xq_hi = at<int8_t>(workspace, L.xq_hi);
        pp.xq_lo = at<uint8_t>(workspace, L.xq_lo);
        pp.xq_s = at<float>(workspace, L.xq_s);
        pp.grp_expert = at<int32_t>(workspace, L.grp_expert);
        pp.grp_off = at<int32_t>(workspace, L.grp_off);
        pp.assign = at<int32_t>(workspace, L.assign);
        if (launch_prep(pp, s, true) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return from_cuda(launch_experts(ep, s));
}

__global__ void set_wait_limit_kernel(WsHeader* h, unsigned long long cycles) { h->wait_limit = cycles; }

}  // namespace

extern "C" {

size_t moe_workspace_bytes(int op, int T, int k, int E, int D, int F) {
    if (T < 1 || k < 1 || E < 1 || D < kBlk || D % kBlk) return 0;
    if (op != MOE_OP_ROUTE && (F < kBlk || F % kBlk)) return 0;
    if (op == MOE_OP_PREFILL) return prefill_shape_ok(E, D, F) ? prefill_layout(T, k, E, D, F).total : 0;
    if (op == MOE_OP_LAYER_RESIDENT) return layer_bytes(T, k, E, D, F) + sizeof(float) * (size_t)T * E;
    if (op == MOE_OP_SHARED) return shared_ws_bytes(T, F);
    if (op == MOE_OP_PREROUTE) return preroute_ws_bytes(T, E, F);
    if (op < MOE_OP_ROUTE || op > MOE_OP_LAYER) return 0;
    if (op == MOE_OP_ROUTE) return layout(op, T, k, E, D, F).total;
    // several tokens through the grouped products (see moe_decode / moe_layer)
    return layer_bytes(T, k, E, D, F);
}

moe_status_t moe_route(const moe_router_t* router, const void* x, moe_dtype_t x_dtype, int T,
                       int32_t* idx, float* w, float* probs, void* workspace, size_t ws_bytes,
                       void* stream) {
    moe_status_t st = check_router(router, x_dtype);
    if (st != MOE_OK) return st;
    if (T < 1 || !al16(x) || !idx || !w) return MOE_ERR_INVALID_ARG;
    Layout L = layout(MOE_OP_ROUTE, T, router->k, router->E, router->D, kBlk);
    if (!workspace || ((uintptr_t)workspace & (kAlign - 1)) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    RouterParams p = router_params(router, x, T, idx, w, probs, workspace, L);
    return from_cuda(launch_router(p, router->w_dtype == MOE_BF16, x_dtype == MOE_BF16,
                                   static_cast<cudaStream_t>(stream), true));
}

moe_status_t moe_substitute(int T, int E, int k, const float* probs, const int32_t* idx_in,
                            const float* w_in, const uint8_t* resident, float threshold,
                            int32_t* idx_out, float* w_out, uint8_t* sub_flag, float* sub_mass,
                            void* stream) {
    if (T < 1 || E < 1 || E > kMaxE || k < 1 || k > kMaxK || k > E) return MOE_ERR_INVALID_ARG;
    if (!probs || !idx_in || !w_in || !resident || !idx_out || !w_out || !sub_flag || !sub_mass)
        return MOE_ERR_INVALID_ARG;
    if (std::isnan(threshold) || threshold < 0.f) return MOE_ERR_INVALID_ARG;
    SubstituteParams p = {T, E, k, probs, idx_in, w_in, resident, threshold, idx_out, w_out, sub_flag, sub_mass};
    return from_cuda(launch_substitute(p, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_decode(const moe_experts_t* experts, const void* x, moe_dtype_t x_dtype, int T,
                        int k, const int32_t* idx, const float* w, float* y, void* x_next,
                        void* workspace, size_t ws_bytes, void* stream) {
    moe_status_t st = check_experts(experts, x_dtype, k);
    if (st != MOE_OK) return st;
    if (T < 1 || T > kMaxDecodeT || !al16(x) || !idx || !w || !al16(y)) return MOE_ERR_INVALID_ARG;
    if (x_next && !al16(x_next)) return MOE_ERR_INVALID_ARG;
    Layout L = layout(MOE_OP_DECODE, T, k, experts->E, experts->D, experts->F);
    if (!workspace || ((uintptr_t)workspace & (kAlign - 1)) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T <= kFusedTokens) {
        FusedCommon fc = fused_common(workspace, L);
        size_t smem = 0;
        int grid = 0;
        if (fused_plan(experts->E, experts->D, experts->F, k, qbits_of(experts), scale_bytes(experts),
                       x_dtype == MOE_BF16 ? 2 : 4, false, &fc, &smem, &grid)) {
            const size_t xb = x_dtype == MOE_BF16 ? 2 : 4;
            for (int t = 0; t < T; t++) {  // one single-token launch per token
                FusedLayer ly = fused_layer(experts, static_cast<const char*>(x) + (size_t)t * experts->D * xb,
                                            y + (size_t)t * experts->D,
                                            x_next ? static_cast<char*>(x_next) + (size_t)t * experts->D * xb
                                                   : nullptr);
                ly.idx_in = idx + (size_t)t * k;
                ly.w_in = w + (size_t)t * k;
                cudaError_t e = launch_fused(fc, &ly, qbits_of(experts), experts->s_dtype == MOE_F16,
                                             x_dtype == MOE_BF16, grid, smem, s);
                if (e != cudaSuccess) return MOE_ERR_CUDA;
            }
            return MOE_OK;
        }
    }
    if (T >= 2 && prefill_shape_ok(experts->E, experts->D, experts->F)) {
        // several tokens: each distinct expert's weights are read once, by the
        // grouped tensor-core products
        PLayout P = prefill_layout(T, k, experts->E, experts->D, experts->F);
        if (ws_bytes < P.total) return MOE_ERR_WORKSPACE;
        return grouped_experts(experts, x, x_dtype, T, k, idx, w, y, x_next, nullptr, nullptr, workspace, P, s);
    }
    ExpertParams ep = expert_params(experts, x, x_dtype, T, k, idx, w, y, x_next, workspace, L);
    PrepParams pp = {};
    pp.T = T;
    pp.E = experts->E;
    pp.D = experts->D;
    pp.k = k;
    pp.qbits = ep.qbits;
    pp.x = x;
    pp.x_bf16 = ep.x_bf16;
    pp.idx = idx;
    pp.hdr = ep.hdr;
    pp.xq_hi = at<int8_t>(workspace, L.xq_hi);
    pp.xq_lo = at<uint8_t>(workspace, L.xq_lo);
    pp.xq_s = at<float>(workspace, L.xq_s);
    pp.grp_expert = at<int32_t>(workspace, L.grp_expert);
    pp.grp_off = at<int32_t>(workspace, L.grp_off);
    pp.assign = at<int32_t>(workspace, L.assign);
    cudaError_t e = launch_prep(pp, s, true);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(launch_experts(ep, s));
}

moe_status_t moe_layer(const moe_router_t* router, const moe_experts_t* experts, const void* x,
                       moe_dtype_t x_dtype, int T, int32_t* idx, float* w, float* probs, float* y,
                       void* x_next, void* workspace, size_t ws_bytes, void* stream) {
    return layer_impl(router, experts, x, x_dtype, T, nullptr, 0.f, idx, w, probs, nullptr, nullptr, nullptr, y,
                      x_next, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_layer_resident(const moe_router_t* router, const moe_experts_t* experts, const void* x,
                                moe_dtype_t x_dtype, int T, const uint8_t* resident, float threshold,
                                int32_t* idx, float* w, float* probs, int32_t* idx_used, uint8_t* sub_flag,
                                float* sub_mass, float* y, void* x_next, void* workspace, size_t ws_bytes,
                                void* stream) {
    if (!resident || !idx_used || !sub_flag || !sub_mass) return MOE_ERR_INVALID_ARG;
    if (std::isnan(threshold) || threshold < 0.f) return MOE_ERR_INVALID_ARG;
    return layer_impl(router, experts, x, x_dtype, T, resident, threshold, idx, w, probs, idx_used, sub_flag,
                      sub_mass, y, x_next, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

// The stacked launch, with or without residency substitution (resident NULL).
static moe_status_t layer_stack_impl(int nlayers, const moe_router_t* routers, const moe_experts_t* experts,
                              const void* const* x, moe_dtype_t x_dtype, int chain, const uint8_t* const* resident,
                              float threshold, int32_t* const* idx, float* const* w, int32_t* const* idx_used,
                              uint8_t* const* sub_flag, float* const* sub_mass, float* const* y,
                              void* const* x_next, void* workspace, size_t ws_bytes, void* stream) {
    if (nlayers < 1 || nlayers > kStackMax || !routers || !experts || !x || !idx || !w || !y)
        return MOE_ERR_INVALID_ARG;
    const moe_router_t& R0 = routers[0];
    const moe_experts_t& X0 = experts[0];
    for (int l = 0; l < nlayers; l++) {
        const moe_router_t& R = routers[l];
        const moe_experts_t& X = experts[l];
        moe_status_t st = check_router(&R, x_dtype);
        if (st != MOE_OK) return st;
        st = check_experts(&X, x_dtype, R.k);
        if (st != MOE_OK) return st;
        if (R.E != X.E || R.D != X.D || R.E != R0.E || R.D != R0.D || R.k != R0.k || R.w_dtype != R0.w_dtype ||
            (R.norm_topk != 0) != (R0.norm_topk != 0) || X.F != X0.F || X.q != X0.q || X.s_dtype != X0.s_dtype)
            return MOE_ERR_INVALID_ARG;
        if ((l == 0 || !chain) && !al16(x[l])) return MOE_ERR_INVALID_ARG;
        if (!idx[l] || !w[l] || !al16(y[l])) return MOE_ERR_INVALID_ARG;
        if (resident && (!resident[l] || !idx_used || !idx_used[l] || !sub_flag || !sub_flag[l] || !sub_mass ||
                         !sub_mass[l]))
            return MOE_ERR_INVALID_ARG;
        void* xn = x_next ? x_next[l] : nullptr;
        if (xn && !al16(xn)) return MOE_ERR_INVALID_ARG;
    }
    if ((R0.w_dtype == MOE_BF16) != (x_dtype == MOE_BF16)) return MOE_ERR_UNSUPPORTED;
    Layout L = layout(MOE_OP_LAYER, 1, R0.k, X0.E, X0.D, X0.F);
    if (!workspace || ((uintptr_t)workspace & (kAlign - 1)) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    FusedCommon fc = fused_common(workspace, L);
    size_t smem = 0;
    int grid = 0;
    if (!fused_plan(X0.E, X0.D, X0.F, R0.k, qbits_of(&X0), scale_bytes(&X0), x_dtype == MOE_BF16 ? 2 : 4, true,
                    &fc, &smem, &grid))
        return MOE_ERR_UNSUPPORTED;
    fc.norm_topk = R0.norm_topk ? 1 : 0;
    fc.threshold = threshold;
    fc.nlayers = nlayers;
    fc.chain = chain ? 1 : 0;
    FusedLayer ly[kStackMax];
    for (int l = 0; l < nlayers; l++) {
        ly[l] = fused_layer(&experts[l], x[l], y[l], x_next ? x_next[l] : nullptr);
        ly[l].W = routers[l].W;
        ly[l].bias = routers[l].bias;
        ly[l].idx = idx[l];
        ly[l].w = w[l];
        if (resident) {
            ly[l].resident = resident[l];
            ly[l].idx_used = idx_used[l];
            ly[l].sub_flag = sub_flag[l];
            ly[l].sub_mass = sub_mass[l];
        }
    }
    return from_cuda(launch_fused(fc, ly, qbits_of(&X0), X0.s_dtype == MOE_F16, x_dtype == MOE_BF16, grid, smem,
                                  static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_stack(int nlayers, const moe_router_t* routers, const moe_experts_t* experts,
                             const void* const* x, moe_dtype_t x_dtype, int chain, int32_t* const* idx,
                             float* const* w, float* const* y, void* const* x_next, void* workspace,
                             size_t ws_bytes, void* stream) {
    return layer_stack_impl(nlayers, routers, experts, x, x_dtype, chain, nullptr, 0.f, idx, w, nullptr, nullptr,
                            nullptr, y, x_next, workspace, ws_bytes, stream);
}

moe_status_t moe_layer_stack_resident(int nlayers, const moe_router_t* routers, const moe_experts_t* experts,
                                      const void* const* x, moe_dtype_t x_dtype, int chain,
                                      const uint8_t* const* resident, float threshold, int32_t* const* idx,
                                      float* const* w, int32_t* const* idx_used, uint8_t* const* sub_flag,
                                      float* const* sub_mass, float* const* y, void* const* x_next, void* workspace,
                                      size_t ws_bytes, void* stream) {
    if (!resident) return MOE_ERR_INVALID_ARG;
    return layer_stack_impl(nlayers, routers, experts, x, x_dtype, chain, resident, threshold, idx, w, idx_used,
                            sub_flag, sub_mass, y, x_next, workspace, ws_bytes, stream);
}

moe_status_t moe_prefill(const moe_router_t* router, const moe_experts_t* experts, const void* x,
                         moe_dtype_t x_dtype, int T, float* y, int32_t* idx, float* w,
                         int32_t* counts, int32_t* perm, void* workspace, size_t ws_bytes,
                         void* stream) {
    moe_status_t st = check_router(router, x_dtype);
    if (st != MOE_OK) return st;
    const int k = router->k;
    st = check_experts(experts, x_dtype, k);
    if (st != MOE_OK) return st;
    if (router->E != experts->E || router->D != experts->D) return MOE_ERR_INVALID_ARG;
    if (T < 1 || !al16(x) || !y) return MOE_ERR_INVALID_ARG;
    const int E = experts->E, D = experts->D, F = experts->F;
    if (!prefill_shape_ok(E, D, F)) return MOE_ERR_UNSUPPORTED;
    PLayout P = prefill_layout(T, k, E, D, F);
    if (!workspace || ((uintptr_t)workspace & (kAlign - 1)) || ws_bytes < P.total) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader* hdr = at<WsHeader>(workspace, 0);
    int32_t* idx_buf = idx ? idx : at<int32_t>(workspace, P.idx);
    float* w_buf = w ? w : at<float>(workspace, P.w);
    float* logits = at<float>(workspace, P.logits);
    moe_status_t rs = route_many(router, x, x_dtype, T, idx_buf, w_buf, nullptr, logits, hdr, s);
    if (rs != MOE_OK) return rs;
    return grouped_experts(experts, x, x_dtype, T, k, idx_buf, w_buf, y, nullptr, counts, perm, workspace, P, s);
}

moe_status_t moe_check_status(void* workspace, void* stream) {
    if (!workspace) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&st, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    // only the status word is cleared: the launch sequence number must keep
    // growing (it tags the values the layer kernel's CTAs exchange), and no
    // kernel leaves a counter behind, even after a wait ran out
    if (st != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return static_cast<moe_status_t>(st);
}

moe_status_t moe_set_wait_limit(void* workspace, unsigned long long cycles, void* stream) {
    if (!workspace || ((uintptr_t)workspace & (kAlign - 1))) return MOE_ERR_WORKSPACE;
    set_wait_limit_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(at<WsHeader>(workspace, 0), cycles);
    return from_cuda(cudaGetLastError());
}

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported combination";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_BAD_INDEX: return "expert id outside [0, E) (access skipped)";
        case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    }
    return "unknown status";
}

}  // extern "C"
