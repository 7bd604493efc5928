// The two parts Edge0 adds around the routed experts (xyznot.com "The Other
// Half of the Memory Wall: Serving 35B MoEs from SSD with Trained Routing
// Prediction", method section):
//
//   moe_shared_lora  the shared expert served with its recovery LoRA left
//                    unmerged ("unmerged adapter execution"): every projection
//                    keeps its quantised base and adds scale * B (A v) beside
//                    it, scale = alpha / r. The adapters sit on the shared
//                    expert, never on the streamed experts.
//   moe_preroute     the prerouter head ("prerouter head architecture"):
//                    logits = fc2 gelu_erf(fc1 f + b1) + L f + bias on
//                    f = [x ; k-hot(current routing) ; k-hot(previous routing)],
//                    then the router's own softmax and top-k, whose ids and
//                    weights are used as the next layer's routing
//                    ("prediction-as-routing").
//
// Both are matrix-vector work for a few tokens, bound by the bytes of their
// weights. One warp owns an output row: it streams the row once with 16-byte
// loads (quantised codes widened in registers, or bf16/fp32 values) and applies
// it to a tile of up to 8 tokens, whose activations come from L2. Kernels of one
// call follow each other on the stream with programmatic dependent launch.
//
// Shared expert, per call (four launches; the adapter launches are skipped
// when r = 0):
//   lora_a_kernel          ax[t] = [A_gate x_t ; A_up x_t]
//   shared_gateup_kernel   h[t][n] = silu(g) * u, g = Gate(x_t)[n] + scale B_gate[n] . ax_gate[t], u likewise
//   lora_a_kernel          ah[t] = A_down h_t
//   shared_down_kernel     y[t][d] (+)= Down(h_t)[d] + scale B_down[d] . ah[t]
// Prerouter, per call (three launches):
//   preroute_hidden_kernel a[t][j] = gelu_erf(fc1[j] . f_t + b1[j])
//   preroute_logits_kernel logits[t][e] = fc2[e] . a_t + L[e] . f_t + bias[e]
//   topk_kernel            fp32 softmax, top-k (lowest id first on equal
//                          probabilities), weights (the router's kernel)
// The k-hot parts of f are never materialised: a row's dot with hot(ids) is
// the sum of the row's entries at the distinct ids that are >= 0.
#include <algorithm>
#include <cmath>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kTokTile = 8;  // tokens one pass over a weight row serves

// 8 consecutive elements (bf16 or fp32) from element e on, widened to fp32 and
// read through L2; e and the base are such that the address is 16-byte aligned.
__device__ __forceinline__ void load8(const void* base, bool bf16, size_t e, float* out) {
    if (bf16) {
        uint4 v = ld_cg16(static_cast<const __nv_bfloat16*>(base) + e);
        out[0] = bf16lo(v.x);
        out[1] = bf16hi(v.x);
        out[2] = bf16lo(v.y);
        out[3] = bf16hi(v.y);
        out[4] = bf16lo(v.z);
        out[5] = bf16hi(v.z);
        out[6] = bf16lo(v.w);
        out[7] = bf16hi(v.w);
    } else {
        const float* p = static_cast<const float*>(base) + e;
        uint4 a = ld_cg16(p), b = ld_cg16(p + 4);
        out[0] = __uint_as_float(a.x);
        out[1] = __uint_as_float(a.y);
        out[2] = __uint_as_float(a.z);
        out[3] = __uint_as_float(a.w);
        out[4] = __uint_as_float(b.x);
        out[5] = __uint_as_float(b.y);
        out[6] = __uint_as_float(b.z);
        out[7] = __uint_as_float(b.w);
    }
}

// One element (bf16 or fp32) through L2.
__device__ __forceinline__ float load1(const void* base, bool bf16, size_t e) {
    return bf16 ? ldcg_f32(static_cast<const __nv_bfloat16*>(base) + e)
                : ldcg_f32(static_cast<const float*>(base) + e);
}

// The signed codes of one 16-byte chunk as floats: 16 int8 codes, or 32 int4
// codes (element 2i in the low nibble of byte i, 2i+1 in the high nibble).
template <int QB>
__device__ __forceinline__ void unpack_chunk(const uint4 w, float* q) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const int b = (int)((u[i >> 2] >> (8 * (i & 3))) & 0xffu);
        if constexpr (QB == 8) {
            q[i] = (float)((b ^ 0x80) - 0x80);
        } else {
            q[2 * i] = (float)(((b & 0xf) ^ 8) - 8);
            q[2 * i + 1] = (float)(((b >> 4) ^ 8) - 8);
        }
    }
}

// Adds this lane's share of sum_k dq(W)[row][k] * v[t][k] to acc[tt] for the
// tokens t = t0 + tt < T. The row has K elements (K a multiple of 32): codes at
// `q` (K or K/2 bytes), scales at `s` (K/32). v is [T][K].
template <int QB, typename ST>
__device__ __forceinline__ void qrow_dot(const uint8_t* q, const ST* s, int K, const void* v, bool v_bf16,
                                         int t0, int T, int lane, float* acc) {
    constexpr int NE = QB == 8 ? 16 : 32;  // elements per 16-byte chunk
    const int nchunk = K / NE;
    for (int c = lane; c < nchunk; c += 32) {
        float wq[NE];
        unpack_chunk<QB>(ld_stream16(q + 16 * c), wq);
        const int e0 = c * NE;
        const float sc = to_f32(s[e0 / kBlk]);
#pragma unroll
        for (int tt = 0; tt < kTokTile; tt++) {
            if (t0 + tt < T) {
                float d = 0.f;
#pragma unroll
                for (int i = 0; i < NE; i += 8) {
                    float xv[8];
                    load8(v, v_bf16, (size_t)(t0 + tt) * K + e0 + i, xv);
#pragma unroll
                    for (int j = 0; j < 8; j++) d = fmaf(wq[i + j], xv[j], d);
                }
                acc[tt] = fmaf(d, sc, acc[tt]);
            }
        }
    }
}

// Adds this lane's share of sum_k W[k] * v[t][k] for a dense bf16/fp32 row of
// K elements (K a multiple of 8) to acc[tt], as qrow_dot.
__device__ __forceinline__ void drow_dot(const void* W, bool w_bf16, size_t row_off, int K, const void* v,
                                         bool v_bf16, size_t ldv, int t0, int T, int lane, float* acc) {
    for (int c = lane; c < K / 8; c += 32) {
        float wv[8];
        load8(W, w_bf16, row_off + 8 * (size_t)c, wv);
#pragma unroll
        for (int tt = 0; tt < kTokTile; tt++) {
            if (t0 + tt < T) {
                float xv[8];
                load8(v, v_bf16, (size_t)(t0 + tt) * ldv + 8 * (size_t)c, xv);
                float d = 0.f;
#pragma unroll
                for (int j = 0; j < 8; j++) d = fmaf(wv[j], xv[j], d);
                acc[tt] += d;
            }
        }
    }
}

// ------------------------------------------------------------ shared expert

struct SharedParams {
    int T, D, F, r;
    int x_bf16, lora_bf16, accumulate;
    float scale;
    const void *gate_q, *gate_s, *up_q, *up_s, *down_q, *down_s;
    const void *gate_B, *up_B, *down_B;
    const void* x;   // [T][D]
    const float* ax; // workspace [T][2r]: A_gate x, A_up x
    float* h;        // workspace [T][F]
    const float* ah; // workspace [T][r]: A_down h
    float* y;        // [T][D]
};

struct LoraAParams {
    int T, K, r, nmat, v_bf16, a_bf16;
    const void* A0;  // [r][K]
    const void* A1;  // [r][K], used when nmat = 2
    const void* v;   // [T][K]
    float* out;      // [T][nmat * r]
};

// out[t][m*r + j] = A_m[j] . v[t]: one warp per output.
__global__ void __launch_bounds__(256) lora_a_kernel(LoraAParams p) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int nout = p.nmat * p.r;
    const long ntask = (long)p.T * nout;
    for (long task = (long)blockIdx.x * 8 + (threadIdx.x >> 5); task < ntask; task += (long)gridDim.x * 8) {
        const int t = (int)(task / nout);
        const int j = (int)(task - (long)t * nout);
        const int m = j / p.r, jj = j - m * p.r;
        float acc[kTokTile] = {};
        // one token: the tile machinery with T = t + 1 and t0 = t
        drow_dot(m ? p.A1 : p.A0, p.a_bf16, (size_t)jj * p.K, p.K, p.v, p.v_bf16, (size_t)p.K, t, t + 1, lane, acc);
        const float s = warp_sum(acc[0]);
        if (lane == 0) p.out[(size_t)t * nout + j] = s;
    }
}

// h[t][n] = silu(Gate(x_t)[n]) * Up(x_t)[n], each projection with its adapter.
template <int QB, typename ST>
__global__ void __launch_bounds__(256) shared_gateup_kernel(SharedParams p) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int rowbytes = QB == 8 ? p.D : p.D / 2;
    const int nb = p.D / kBlk;
    const uint8_t* GQ = static_cast<const uint8_t*>(p.gate_q);
    const uint8_t* UQ = static_cast<const uint8_t*>(p.up_q);
    const ST* GS = static_cast<const ST*>(p.gate_s);
    const ST* US = static_cast<const ST*>(p.up_s);
    for (int n = blockIdx.x * 8 + (threadIdx.x >> 5); n < p.F; n += gridDim.x * 8) {
        for (int t0 = 0; t0 < p.T; t0 += kTokTile) {
            float ag[kTokTile] = {}, au[kTokTile] = {};
            qrow_dot<QB, ST>(GQ + (size_t)n * rowbytes, GS + (size_t)n * nb, p.D, p.x, p.x_bf16, t0, p.T, lane, ag);
            qrow_dot<QB, ST>(UQ + (size_t)n * rowbytes, US + (size_t)n * nb, p.D, p.x, p.x_bf16, t0, p.T, lane, au);
            for (int j = lane; j < p.r; j += 32) {
                const float bg = p.scale * load1(p.gate_B, p.lora_bf16, (size_t)n * p.r + j);
                const float bu = p.scale * load1(p.up_B, p.lora_bf16, (size_t)n * p.r + j);
#pragma unroll
                for (int tt = 0; tt < kTokTile; tt++) {
                    if (t0 + tt < p.T) {
                        const float* axt = p.ax + (size_t)(t0 + tt) * 2 * p.r;
                        ag[tt] = fmaf(bg, ld_cg_f32(axt + j), ag[tt]);
                        au[tt] = fmaf(bu, ld_cg_f32(axt + p.r + j), au[tt]);
                    }
                }
            }
#pragma unroll
            for (int tt = 0; tt < kTokTile; tt++) {
                if (t0 + tt < p.T) {
                    const float g = warp_sum(ag[tt]), u = warp_sum(au[tt]);
                    if (lane == 0) p.h[(size_t)(t0 + tt) * p.F + n] = silu_mul(g, u);
                }
            }
        }
    }
}

// y[t][d] (+)= Down(h_t)[d] with its adapter.
template <int QB, typename ST>
__global__ void __launch_bounds__(256) shared_down_kernel(SharedParams p) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int rowbytes = QB == 8 ? p.F : p.F / 2;
    const int nb = p.F / kBlk;
    const uint8_t* DQ = static_cast<const uint8_t*>(p.down_q);
    const ST* DS = static_cast<const ST*>(p.down_s);
    for (int d = blockIdx.x * 8 + (threadIdx.x >> 5); d < p.D; d += gridDim.x * 8) {
        for (int t0 = 0; t0 < p.T; t0 += kTokTile) {
            float acc[kTokTile] = {};
            qrow_dot<QB, ST>(DQ + (size_t)d * rowbytes, DS + (size_t)d * nb, p.F, p.h, false, t0, p.T, lane, acc);
            for (int j = lane; j < p.r; j += 32) {
                const float b = p.scale * load1(p.down_B, p.lora_bf16, (size_t)d * p.r + j);
#pragma unroll
                for (int tt = 0; tt < kTokTile; tt++)
                    if (t0 + tt < p.T) acc[tt] = fmaf(b, ld_cg_f32(p.ah + (size_t)(t0 + tt) * p.r + j), acc[tt]);
            }
#pragma unroll
            for (int tt = 0; tt < kTokTile; tt++) {
                if (t0 + tt < p.T) {
                    const float o = warp_sum(acc[tt]);
                    if (lane == 0) {
                        float* yo = p.y + (size_t)(t0 + tt) * p.D + d;
                        *yo = p.accumulate ? ld_cg_f32(yo) + o : o;
                    }
                }
            }
        }
    }
}

// --------------------------------------------------------------- prerouter

struct PrerouteParams {
    int T, D, E, H, k;
    int w_bf16, x_bf16;
    const void* x;          // [T][D]
    const int32_t* cur;     // [T][k]
    const int32_t* prev;    // [T][k]
    const void* fc1;        // [H][D+2E]
    const float* b1;        // [H] or null
    const void* fc2;        // [E][H]
    const void* L;          // [E][D+2E]
    const float* bias;      // [E] or null
    float* a;               // workspace [T][H]
    float* logits;          // workspace [T][E]
    WsHeader* hdr;
};

// This lane's share of a row's dot with [hot(cur[t]) ; hot(prev[t])]: the
// row's entries D + id (current) and D + E + id (previous) over the distinct
// ids >= 0 of the token's lists. An id >= E is recorded and skipped.
__device__ __forceinline__ float hot_dot(const PrerouteParams& p, const void* W, size_t row_off, int t, int lane) {
    float acc = 0.f;
    for (int i = lane; i < 2 * p.k; i += 32) {
        const bool is_prev = i >= p.k;
        const int r = is_prev ? i - p.k : i;
        const int32_t* ids = (is_prev ? p.prev : p.cur) + (size_t)t * p.k;
        const int e = ld_cg_i32(ids + r);
        if (e < 0) continue;
        if (e >= p.E) {
            record_error(&p.hdr->status, MOE_ERR_BAD_INDEX);
            continue;
        }
        bool repeat = false;
        for (int r2 = 0; r2 < r; r2++) repeat |= ld_cg_i32(ids + r2) == e;
        if (repeat) continue;
        acc += load1(W, p.w_bf16, row_off + (size_t)p.D + (is_prev ? (size_t)p.E : 0) + e);
    }
    return acc;
}

__global__ void __launch_bounds__(256) preroute_hidden_kernel(PrerouteParams p) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const size_t nf = (size_t)p.D + 2 * (size_t)p.E;
    for (int j = blockIdx.x * 8 + (threadIdx.x >> 5); j < p.H; j += gridDim.x * 8) {
        for (int t0 = 0; t0 < p.T; t0 += kTokTile) {
            float acc[kTokTile] = {};
            drow_dot(p.fc1, p.w_bf16, (size_t)j * nf, p.D, p.x, p.x_bf16, (size_t)p.D, t0, p.T, lane, acc);
#pragma unroll
            for (int tt = 0; tt < kTokTile; tt++) {
                if (t0 + tt < p.T) {
                    const float z = warp_sum(acc[tt] + hot_dot(p, p.fc1, (size_t)j * nf, t0 + tt, lane)) +
                                    (p.b1 ? p.b1[j] : 0.f);
                    if (lane == 0) p.a[(size_t)(t0 + tt) * p.H + j] = 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
                }
            }
        }
    }
}

__global__ void __launch_bounds__(256) preroute_logits_kernel(PrerouteParams p) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const size_t nf = (size_t)p.D + 2 * (size_t)p.E;
    for (int e = blockIdx.x * 8 + (threadIdx.x >> 5); e < p.E; e += gridDim.x * 8) {
        for (int t0 = 0; t0 < p.T; t0 += kTokTile) {
            float acc[kTokTile] = {};
            drow_dot(p.L, p.w_bf16, (size_t)e * nf, p.D, p.x, p.x_bf16, (size_t)p.D, t0, p.T, lane, acc);
            drow_dot(p.fc2, p.w_bf16, (size_t)e * p.H, p.H, p.a, false, (size_t)p.H, t0, p.T, lane, acc);
#pragma unroll
            for (int tt = 0; tt < kTokTile; tt++) {
                if (t0 + tt < p.T) {
                    const float z = warp_sum(acc[tt] + hot_dot(p, p.L, (size_t)e * nf, t0 + tt, lane)) +
                                    (p.bias ? p.bias[e] : 0.f);
                    if (lane == 0) p.logits[(size_t)(t0 + tt) * p.E + e] = z;
                }
            }
        }
    }
}

// ---------------------------------------------------------------- host side

constexpr size_t kWsAlign = 256;
constexpr int kMaxRank = 64;
constexpr int kMaxRows = 152 * 8;  // CTAs of a row kernel; more rows loop

size_t up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }
bool al16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }
unsigned row_grid(long rows) { return (unsigned)std::max(1L, std::min((long)kMaxRows, (rows + 7) / 8)); }

struct SharedLayout {
    size_t ax, h, ah, total;
};
SharedLayout shared_layout(int T, int F) {
    SharedLayout L;
    size_t o = sizeof(WsHeader);
    L.ax = o;
    o += up(sizeof(float) * (size_t)T * 2 * kMaxRank);
    L.h = o;
    o += up(sizeof(float) * (size_t)T * F);
    L.ah = o;
    o += up(sizeof(float) * (size_t)T * kMaxRank);
    L.total = o;
    return L;
}

struct PrerouteLayout {
    size_t a, logits, total;
};
PrerouteLayout preroute_layout(int T, int E, int H) {
    PrerouteLayout L;
    size_t o = sizeof(WsHeader);
    L.a = o;
    o += up(sizeof(float) * (size_t)T * H);
    L.logits = o;
    o += up(sizeof(float) * (size_t)T * E);
    L.total = o;
    return L;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

size_t shared_ws_bytes(int T, int F) { return shared_layout(T, F).total; }
size_t preroute_ws_bytes(int T, int E, int H) { return preroute_layout(T, E, H).total; }

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_shared_lora(const moe_shared_t* se, const void* x, moe_dtype_t x_dtype, int T,
                                        float* y, int accumulate, void* workspace, size_t ws_bytes,
                                        void* stream) {
    if (!se) return MOE_ERR_INVALID_ARG;
    const int D = se->D, F = se->F, r = se->r;
    if (T < 1 || D < kBlk || D % kBlk || F < kBlk || F % kBlk || r < 0 || r > kMaxRank) return MOE_ERR_INVALID_ARG;
    if (se->q != MOE_Q_INT8_SYM_B32 && se->q != MOE_Q_INT4_SYM_B32) return MOE_ERR_UNSUPPORTED;
    if (se->s_dtype != MOE_F32 && se->s_dtype != MOE_F16) return MOE_ERR_UNSUPPORTED;
    if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    const void* base[6] = {se->gate_q, se->gate_s, se->up_q, se->up_s, se->down_q, se->down_s};
    for (const void* p : base)
        if (!al16(p)) return MOE_ERR_INVALID_ARG;
    if (!al16(x) || !al16(y)) return MOE_ERR_INVALID_ARG;
    if (r > 0) {
        if (se->lora_dtype != MOE_F32 && se->lora_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
        const void* ad[6] = {se->gate_A, se->gate_B, se->up_A, se->up_B, se->down_A, se->down_B};
        for (const void* p : ad)
            if (!al16(p)) return MOE_ERR_INVALID_ARG;
        if (!std::isfinite(se->lora_scale)) return MOE_ERR_INVALID_ARG;
    }
    const SharedLayout L = shared_layout(T, F);
    if (!workspace || ((uintptr_t)workspace & (kWsAlign - 1)) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;

    SharedParams p = {};
    p.T = T;
    p.D = D;
    p.F = F;
    p.r = r;
    p.x_bf16 = x_dtype == MOE_BF16;
    p.lora_bf16 = se->lora_dtype == MOE_BF16;
    p.accumulate = accumulate ? 1 : 0;
    p.scale = r > 0 ? se->lora_scale : 0.f;
    p.gate_q = se->gate_q;
    p.gate_s = se->gate_s;
    p.up_q = se->up_q;
    p.up_s = se->up_s;
    p.down_q = se->down_q;
    p.down_s = se->down_s;
    p.gate_B = se->gate_B;
    p.up_B = se->up_B;
    p.down_B = se->down_B;
    p.x = x;
    p.ax = at<float>(workspace, L.ax);
    p.h = at<float>(workspace, L.h);
    p.ah = at<float>(workspace, L.ah);
    p.y = y;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool q8 = se->q == MOE_Q_INT8_SYM_B32, f16 = se->s_dtype == MOE_F16;
    const unsigned ga = row_grid(F), gd = row_grid(D);
    cudaError_t e = cudaSuccess;
    if (r > 0) {
        LoraAParams la = {T, D, r, 2, p.x_bf16, p.lora_bf16, se->gate_A, se->up_A, x, at<float>(workspace, L.ax)};
        e = launch(lora_a_kernel, dim3(row_grid((long)T * 2 * r)), dim3(256), 0, s, true, la);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (q8)
        e = f16 ? launch(shared_gateup_kernel<8, __half>, dim3(ga), dim3(256), 0, s, true, p)
                : launch(shared_gateup_kernel<8, float>, dim3(ga), dim3(256), 0, s, true, p);
    else
        e = f16 ? launch(shared_gateup_kernel<4, __half>, dim3(ga), dim3(256), 0, s, true, p)
                : launch(shared_gateup_kernel<4, float>, dim3(ga), dim3(256), 0, s, true, p);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (r > 0) {
        LoraAParams la = {T, F, r, 1, 0, p.lora_bf16, se->down_A, nullptr, p.h, at<float>(workspace, L.ah)};
        e = launch(lora_a_kernel, dim3(row_grid((long)T * r)), dim3(256), 0, s, true, la);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (q8)
        e = f16 ? launch(shared_down_kernel<8, __half>, dim3(gd), dim3(256), 0, s, true, p)
                : launch(shared_down_kernel<8, float>, dim3(gd), dim3(256), 0, s, true, p);
    else
        e = f16 ? launch(shared_down_kernel<4, __half>, dim3(gd), dim3(256), 0, s, true, p)
                : launch(shared_down_kernel<4, float>, dim3(gd), dim3(256), 0, s, true, p);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_preroute(const moe_prerouter_t* head, const void* x, moe_dtype_t x_dtype, int T,
                                     const int32_t* cur, const int32_t* prev, int32_t* idx, float* w,
                                     float* probs, void* workspace, size_t ws_bytes, void* stream) {
    if (!head) return MOE_ERR_INVALID_ARG;
    const int D = head->D, E = head->E, H = head->H, k = head->k;
    if (T < 1 || D < kBlk || D % kBlk || H < kBlk || H % kBlk) return MOE_ERR_INVALID_ARG;
    if (E < 4 || E % 4 || E > 1024 || k < 1 || k > 32 || k > E) return MOE_ERR_INVALID_ARG;
    if (head->w_dtype != MOE_F32 && head->w_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (!al16(head->fc1) || !al16(head->fc2) || !al16(head->L) || !al16(x)) return MOE_ERR_INVALID_ARG;
    if ((head->b1 && ((uintptr_t)head->b1 & 3u)) || (head->bias && ((uintptr_t)head->bias & 3u)))
        return MOE_ERR_INVALID_ARG;
    if (!cur || !prev || !idx || !w) return MOE_ERR_INVALID_ARG;
    const PrerouteLayout L = preroute_layout(T, E, H);
    if (!workspace || ((uintptr_t)workspace & (kWsAlign - 1)) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;

    PrerouteParams p = {};
    p.T = T;
    p.D = D;
    p.E = E;
    p.H = H;
    p.k = k;
    p.w_bf16 = head->w_dtype == MOE_BF16;
    p.x_bf16 = x_dtype == MOE_BF16;
    p.x = x;
    p.cur = cur;
    p.prev = prev;
    p.fc1 = head->fc1;
    p.b1 = head->b1;
    p.fc2 = head->fc2;
    p.L = head->L;
    p.bias = head->bias;
    p.a = at<float>(workspace, L.a);
    p.logits = at<float>(workspace, L.logits);
    p.hdr = at<WsHeader>(workspace, 0);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch(preroute_hidden_kernel, dim3(row_grid(H)), dim3(256), 0, s, true, p);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = launch(preroute_logits_kernel, dim3(row_grid(E)), dim3(256), 0, s, true, p);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    TopkParams tp = {T, E, k, head->norm_topk ? 1 : 0, p.logits, nullptr, idx, w, probs};
    return launch_topk(tp, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
