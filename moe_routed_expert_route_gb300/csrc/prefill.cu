// Grouping and routing for many tokens (prefill, and decode of T >= 2):
// router logits on the tensor cores, the warp top-k, the stable grouping of the
// (token, slot) assignments by expert, the scaled fp16 gather of x in grouped
// order and the weighted un-permute. The expert products themselves are in
// egemm.cu. Kernels, in stream order:
//   router_gemm  logits = X Wr^T on the tensor cores (bf16 x bf16 -> fp32)
//   topk         bias, fp32 softmax and top-k per token (one warp per token)
//   hist/scan/place  stable counting sort of the T*k assignments by expert:
//                per-chunk histograms, one scan (offsets, per-chunk bases and
//                the list of token tiles per expert), then placement in (t, r)
//                order inside every expert
//   gather_f16   x rows in grouped order, fp16, one power-of-two scale per row
//   (egemm gate/up with SwiGLU, egemm down)
//   combine      y[t] = sum_r w[t][r] * Y[inv[t][r]], slot order fixed, and
//                x_next = x + y
//
// The router product (one CTA per 128 x 128 tile of logits): one thread
// streams the x and Wr tiles by TMA (128-byte swizzle, 4 stages of 64 along
// K), one thread issues tcgen05.mma.cta_group::1.kind::f16 (bf16, M = N = 128,
// K = 16) into a 128-column TMEM accumulator and commits to per-stage
// mbarriers; four warps read TMEM with tcgen05.ld for the fp32 epilogue.
// Every wait is bounded.
#include <mutex>

#include "group.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

constexpr int kGM = 128;   // tile rows (tokens)
constexpr int kGN = 128;   // tile columns (experts)
constexpr int kGK = 64;    // K per stage = one 128-byte row of 16-bit values
constexpr int kGS = 4;     // stages
constexpr int kGThreads = 224;
constexpr size_t kGSmem = (size_t)kGS * 2 * 16384 + 1024;  // A + B tile per stage, 1 KB alignment

// Roles (7 warps): warp 6 streams both tiles by TMA, one thread of warp 5
// issues the MMAs and owns the TMEM allocation, warps 1-4 run the epilogue
// (TMEM lane quarter = warp % 4).
__global__ void __launch_bounds__(kGThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ unsigned char sm_raw[];
    unsigned char* ab = reinterpret_cast<unsigned char*>(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t a_full[kGS], ab_empty[kGS], done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x / p.n_ntiles, nt = blockIdx.x - (blockIdx.x / p.n_ntiles) * p.n_ntiles;
    pdl_wait();
    pdl_trigger();
    if (mt >= p.n_mtiles) return;  // whole CTA, before any barrier or allocation
    const int m0 = mt * kGM;
    const int nk = p.K / kGK;
    int* status = &p.hdr->status;

    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kGS; i++) {
            mbar_init(&a_full[i], 1);
            mbar_init(&ab_empty[i], 1);
        }
        mbar_init(&done, 1);
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(&s_tmem, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int brow0 = nt * p.rows_per_ntile;

    if (warp == 6) {
        // ------------------------------------------------ A and B producer
        if (lane == 0) {
            for (int t = 0; t < nk; t++) {
                const int s = t % kGS;
                if (t >= kGS && !mbar_wait(&ab_empty[s], ((t / kGS) - 1) & 1, status)) {
                    s_abort = 1;
                    break;
                }
                unsigned char* dst = ab + (size_t)s * 32768;
                mbar_arrive_expect_tx(&a_full[s], 32768);
                tma_load_2d(dst, &p.tmA, t * kGK, m0, &a_full[s]);
                tma_load_2d(dst + 16384, &p.tmB0, t * kGK, brow0, &a_full[s]);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_f16(true, kGM, kGN);
            for (int t = 0; t < nk; t++) {
                const int s = t % kGS;
                if (s_abort || !mbar_wait(&a_full[s], (t / kGS) & 1, status)) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_addr(ab + (size_t)s * 32768);
                const uint64_t ad = umma_desc_sw128(a0), bd = umma_desc_sw128(a0 + 16384);
#pragma unroll
                for (int kk = 0; kk < kGK / 16; kk++)
                    umma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (t | kk) != 0 ? 1u : 0u);
                umma_commit(&ab_empty[s]);
            }
            umma_commit(&done);  // also after an abort: completes when the issued MMAs are done
        }
    } else if (warp >= 1 && warp <= 4) {
        // ------------------------------------------------ epilogue
        if (!mbar_wait(&done, 0, status)) s_abort = 1;
        tc_fence_after();
        const int row = 32 * (warp & 3) + lane;  // TMEM lane quarter of this warp
        const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const int pos = m0 + row;
        const bool valid = pos < p.m_total && !s_abort;
        float* C = reinterpret_cast<float*>(p.C) + (size_t)pos * p.ldc + nt * kGN;
#pragma unroll
        for (int c = 0; c < 8; c++) {
            uint32_t v[16];
            tmem_ld16(trow + 16 * c, v);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
                for (int q = 0; q < 4; q++)
                    reinterpret_cast<uint4*>(C + 16 * c)[q] =
                        make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) tmem_dealloc(tmem, 128);
}

cudaError_t launch_router_gemm(const GemmParams& p, cudaStream_t s) {
    return launch(gemm_tc_kernel, dim3(p.n_mtiles * p.n_ntiles), dim3(kGThreads), kGSmem, s, true, p);
}

// ---------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// The encoded maps of recent calls, keyed by every argument of the encoding
// (a map depends on nothing else), so that a layer called again with the same
// buffers does not pay the driver's encoding on every call.
namespace {
struct TmapKey {
    const void* base;
    unsigned long long inner, rows, row_bytes;
    unsigned box_inner, box_rows;
    int dtype, swizzle;
    bool operator==(const TmapKey& o) const {
        return base == o.base && inner == o.inner && rows == o.rows && row_bytes == o.row_bytes &&
               box_inner == o.box_inner && box_rows == o.box_rows && dtype == o.dtype && swizzle == o.swizzle;
    }
};
constexpr int kTmapCache = 64;
struct TmapCache {
    std::mutex mu;
    TmapKey key[kTmapCache];
    CUtensorMap map[kTmapCache];
    int n = 0, next = 0;
};
TmapCache& tmap_cache() {
    static TmapCache c;
    return c;
}
}  // namespace

static bool encode_tmap_2d(CUtensorMap* m, int dtype, const void* base, unsigned long long inner,
                           unsigned long long rows, unsigned long long row_bytes, unsigned box_inner,
                           unsigned box_rows, int swizzle);

bool make_tmap_2d(CUtensorMap* m, int dtype, const void* base, unsigned long long inner, unsigned long long rows,
                  unsigned long long row_bytes, unsigned box_inner, unsigned box_rows, int swizzle) {
    const TmapKey k = {base, inner, rows, row_bytes, box_inner, box_rows, dtype, swizzle};
    TmapCache& c = tmap_cache();
    {
        std::lock_guard<std::mutex> lock(c.mu);
        for (int i = 0; i < c.n; i++)
            if (c.key[i] == k) {
                *m = c.map[i];
                return true;
            }
    }
    if (!encode_tmap_2d(m, dtype, base, inner, rows, row_bytes, box_inner, box_rows, swizzle)) return false;
    std::lock_guard<std::mutex> lock(c.mu);
    const int i = c.n < kTmapCache ? c.n++ : c.next;
    c.next = (i + 1) % kTmapCache;
    c.key[i] = k;
    c.map[i] = *m;
    return true;
}

static bool encode_tmap_2d(CUtensorMap* m, int dtype, const void* base, unsigned long long inner,
                           unsigned long long rows, unsigned long long row_bytes, unsigned box_inner,
                           unsigned box_rows, int swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUtensorMapDataType dt = dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                            : dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMapSwizzle sw = swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                          : swizzle == 32  ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE;
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// x rows in grouped order as fp16, each scaled by a power of two so that its
// largest magnitude lies in (1/2, 1]: Xp[pos] = fp16(x[t] * 2^-e), t =
// perm_tok[pos], e = pexp[pos]. Scaling by 2^-e is exact, and fp16 keeps its
// relative precision at any scale, so this only keeps rows whose values exceed
// the fp16 range (a residual stream that has grown) finite; the products undo
// it exactly in their epilogues. One CTA per position.
__global__ void __launch_bounds__(256) gather_f16_kernel(const void* x, int x_bf16, const int32_t* perm_tok,
                                                         int n, int D, __half* Xp, int32_t* pexp) {
    constexpr int kV = 4;  // 8-element vectors per thread (D <= 8192)
    __shared__ float s_m[8];
    pdl_wait();
    pdl_trigger();
    const int pos = blockIdx.x, tid = threadIdx.x;
    if (pos >= n) return;
    const int t = ld_cg_i32(perm_tok + pos);
    const int nv = D / 8;
    float f[kV][8];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < kV; i++) {
        const int v = tid + 256 * i;
#pragma unroll
        for (int q = 0; q < 8; q++) f[i][q] = 0.f;
        if (v < nv) {
            if (x_bf16) load_f32_cg<__nv_bfloat16, 8>(reinterpret_cast<const __nv_bfloat16*>(x) + (size_t)t * D + 8 * v, f[i]);
            else load_f32_cg<float, 8>(reinterpret_cast<const float*>(x) + (size_t)t * D + 8 * v, f[i]);
        }
#pragma unroll
        for (int q = 0; q < 8; q++) m = fmaxf(m, fabsf(f[i][q]));
    }
    m = warp_max(m);
    if ((tid & 31) == 0) s_m[tid >> 5] = m;
    __syncthreads();
    m = s_m[0];
#pragma unroll
    for (int i = 1; i < 8; i++) m = fmaxf(m, s_m[i]);
    // e with m * 2^-e in (1/2, 1] (0 for a zero or non-finite row)
    int e = 0;
    if (m > 0.f && m <= 3.0e38f) {
        e = ((__float_as_int(m) >> 23) & 0xff) - 126;
        if ((__float_as_int(m) & 0x7fffff) == 0) e -= 1;  // m a power of two: m * 2^-e = 1
        e = max(-60, min(60, e));  // 2^(2e) stays a normal fp32 factor
    }
    const float sc = __int_as_float((127 - e) << 23);  // 2^-e
    if (tid == 0) pexp[pos] = e;
#pragma unroll
    for (int i = 0; i < kV; i++) {
        const int v = tid + 256 * i;
        if (v < nv) {
            uint4 o;
            uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                __half2 h = __floats2half2_rn(f[i][2 * q] * sc, f[i][2 * q + 1] * sc);
                ow[q] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(Xp + (size_t)pos * D + 8 * v) = o;
        }
    }
}

cudaError_t launch_gather_f16(const void* x, bool x_bf16, const int32_t* perm_tok, int n, int D, void* Xp,
                              int32_t* pexp, cudaStream_t s) {
    return launch(gather_f16_kernel, dim3((unsigned)std::max(n, 1)), dim3(256), 0, s, true, x, x_bf16 ? 1 : 0,
                  perm_tok, n, D, reinterpret_cast<__half*>(Xp), pexp);
}

// ----------------------------------------------------------- routing

// logits (+ bias) -> fp32 softmax -> top-k, one warp per token.
template <int NJ>
__global__ void __launch_bounds__(256) topk_kernel(TopkParams p) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    __shared__ uint64_t s_tk[8][kTopkScratch];
    pdl_wait();
    pdl_trigger();
    if (t >= p.T) return;
    float v[NJ];
#pragma unroll
    for (int j = 0; j < NJ; j++) {
        int e = j * 32 + lane;
        v[j] = e < p.E ? ld_cg_f32(p.logits + (size_t)t * p.E + e) + (p.bias ? p.bias[e] : 0.f) : 0.f;
    }
    int sel_e;
    float sel_p;
    softmax_topk_regs<NJ>(v, p.E, p.k, p.probs ? p.probs + (size_t)t * p.E : nullptr, lane, s_tk[threadIdx.x >> 5],
                          sel_e, sel_p);
    float norm = warp_sum(lane < p.k ? sel_p : 0.f);
    if (lane < p.k) {
        p.idx[(size_t)t * p.k + lane] = sel_e;
        p.w[(size_t)t * p.k + lane] = p.norm_topk ? sel_p / norm : sel_p;
    }
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s) {
    dim3 grid((p.T + 7) / 8), block(256);
    switch (topk_nj(p.E, p.k)) {
        case 1: return launch(topk_kernel<1>, grid, block, 0, s, true, p);
        case 2: return launch(topk_kernel<2>, grid, block, 0, s, true, p);
        case 4: return launch(topk_kernel<4>, grid, block, 0, s, true, p);
        case 8: return launch(topk_kernel<8>, grid, block, 0, s, true, p);
        case 16: return launch(topk_kernel<16>, grid, block, 0, s, true, p);
        default: return launch(topk_kernel<32>, grid, block, 0, s, true, p);
    }
}

// ------------------------------------------------------ grouping by expert

// Per-chunk histograms of expert ids (chunk = kPermChunk assignments).
__global__ void __launch_bounds__(256) perm_hist_kernel(PermParams p) {
    extern __shared__ int s_cnt[];
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    const int i0 = c * kPermChunk, i1 = min(p.n, i0 + kPermChunk);
    for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
        int e = ld_cg_i32(p.idx + i);
        if (e >= 0 && e < p.E) atomicAdd(&s_cnt[e], 1);
        else record_error(&p.hdr->status, MOE_ERR_BAD_INDEX);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) p.chunk_cnt[(size_t)c * p.E + e] = s_cnt[e];
}

// One CTA: totals, exclusive offsets, per-chunk bases, and the tile list.
__global__ void __launch_bounds__(1024) perm_scan_kernel(PermParams p) {
    __shared__ int s_w1[32], s_w2[32];
    pdl_wait();
    pdl_trigger();
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    int cnt = 0;
    if (e < p.E)
        for (int c = 0; c < p.nchunk; c++) cnt += ld_cg_i32(p.chunk_cnt + (size_t)c * p.E + e);
    const int tiles = (cnt + p.tile_rows - 1) / p.tile_rows;
    // block exclusive scan of (cnt, tiles) over e
    int a = cnt, b = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int x = __shfl_up_sync(kFull, a, o), y = __shfl_up_sync(kFull, b, o);
        if (lane >= o) { a += x; b += y; }
    }
    if (lane == 31) { s_w1[warp] = a; s_w2[warp] = b; }
    __syncthreads();
    if (warp == 0) {
        int x = s_w1[lane], y = s_w2[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int xx = __shfl_up_sync(kFull, x, o), yy = __shfl_up_sync(kFull, y, o);
            if (lane >= o) { x += xx; y += yy; }
        }
        s_w1[lane] = x;
        s_w2[lane] = y;
    }
    __syncthreads();
    const int off = a - cnt + (warp ? s_w1[warp - 1] : 0);
    const int toff = b - tiles + (warp ? s_w2[warp - 1] : 0);
    if (e < p.E) {
        p.cnt[e] = cnt;
        p.off[e] = off;
        p.group_end[e] = off + cnt;
        if (p.counts_out) p.counts_out[e] = cnt;
        int base = off;
        for (int c = 0; c < p.nchunk; c++) {
            p.chunk_base[(size_t)c * p.E + e] = base;
            base += ld_cg_i32(p.chunk_cnt + (size_t)c * p.E + e);
        }
        for (int i = 0; i < tiles; i++) {
            p.tile_group[toff + i] = e;
            p.tile_m0[toff + i] = off + i * p.tile_rows;
            if (p.tile_n) p.tile_n[toff + i] = min(p.tile_rows, cnt - i * p.tile_rows);
        }
        if (e == p.E - 1) {
            p.off[p.E] = off + cnt;
            *p.n_mtiles = toff + tiles;
        }
    }
}

// Stable placement: assignments of a chunk in (t, r) order, 32 at a time.
__global__ void __launch_bounds__(32) perm_place_kernel(PermParams p) {
    extern __shared__ int s_run[];
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x, lane = threadIdx.x;
    for (int e = lane; e < p.E; e += 32) s_run[e] = ld_cg_i32(p.chunk_base + (size_t)c * p.E + e);
    __syncwarp();
    const int i0 = c * kPermChunk, i1 = min(p.n, i0 + kPermChunk);
    const unsigned lt = (1u << lane) - 1u;
    for (int base = i0; base < i1; base += 32) {
        const int i = base + lane;
        int e = i < i1 ? ld_cg_i32(p.idx + i) : -1;
        const bool ok = e >= 0 && e < p.E;
        const unsigned peers = __match_any_sync(kFull, ok ? e : -2 - lane);
        const int rank = __popc(peers & lt);
        const int pos = ok ? s_run[e] + rank : 0;
        __syncwarp();
        if (ok) {
            if (rank == 0) s_run[e] += __popc(peers);
            p.perm_tok[pos] = i / p.k;
            if (p.perm_out) p.perm_out[pos] = i;
            p.inv[i] = pos;
        } else if (i < i1) {
            p.inv[i] = -1;
        }
        __syncwarp();
    }
}

cudaError_t launch_perm(const PermParams& p, cudaStream_t s) {
    cudaError_t e = launch(perm_hist_kernel, dim3(p.nchunk), dim3(256), sizeof(int) * p.E, s, true, p);
    if (e != cudaSuccess) return e;
    e = launch(perm_scan_kernel, dim3(1), dim3(1024), 0, s, true, p);
    if (e != cudaSuccess) return e;
    return launch(perm_place_kernel, dim3(p.nchunk), dim3(32), sizeof(int) * p.E, s, true, p);
}

// ------------------------------------------------------------- combine
// y[t][d] = sum_r w[t][r] * Y[inv[t][r]][d], r = 0, 1, ..., k-1; 4 d per thread.
__global__ void __launch_bounds__(256) combine_kernel(CombineParams p) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.y;
    const int d = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (t >= p.T || d >= p.D) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < p.k; r++) {
        const int pos = ld_cg_i32(p.inv + (size_t)t * p.k + r);
        if (pos < 0) continue;
        const float w = ld_cg_f32(p.w + (size_t)t * p.k + r);
        uint4 v = ld_cg16(p.Y + (size_t)pos * p.D + d);
        acc.x = fmaf(w, __uint_as_float(v.x), acc.x);
        acc.y = fmaf(w, __uint_as_float(v.y), acc.y);
        acc.z = fmaf(w, __uint_as_float(v.z), acc.z);
        acc.w = fmaf(w, __uint_as_float(v.w), acc.w);
    }
    *reinterpret_cast<float4*>(p.y + (size_t)t * p.D + d) = acc;
    if (p.x_next) {
        const size_t o = (size_t)t * p.D + d;
        if (p.x_bf16) {
            float xv[4];
            load_f32_cg<__nv_bfloat16, 4>(reinterpret_cast<const __nv_bfloat16*>(p.x) + o, xv);
            __nv_bfloat16* xn = reinterpret_cast<__nv_bfloat16*>(p.x_next) + o;
            xn[0] = __float2bfloat16_rn(xv[0] + acc.x);
            xn[1] = __float2bfloat16_rn(xv[1] + acc.y);
            xn[2] = __float2bfloat16_rn(xv[2] + acc.z);
            xn[3] = __float2bfloat16_rn(xv[3] + acc.w);
        } else {
            const float4 xv = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.x) + o);
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.x_next) + o) =
                make_float4(xv.x + acc.x, xv.y + acc.y, xv.z + acc.z, xv.w + acc.w);
        }
    }
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
    dim3 grid((p.D / 4 + 255) / 256, p.T), block(256);
    return launch(combine_kernel, grid, block, 0, s, true, p);
}

}  // namespace moe
