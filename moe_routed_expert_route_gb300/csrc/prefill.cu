// Prefill of many tokens: routing, grouping of the (token, slot) assignments
// by expert, one grouped matrix product per projection on the 5th-generation
// tensor cores, and the weighted un-permute.
//
// With thousands of tokens every routed expert serves a batch of tokens, so
// its projections are dense contractions: X_e [m_e x D] times the expert's
// dequantised weights. Kernels, in stream order:
//   router_gemm  logits = X Wr^T on the tensor cores (bf16 x bf16 -> fp32)
//   topk         bias, fp32 softmax and top-k per token (one warp per token)
//   to_f16       x -> fp16 copy (the A operand of the expert products)
//   hist/scan/place  stable counting sort of the T*k assignments by expert:
//                per-chunk histograms, one scan (offsets, per-chunk bases and
//                the list of 128-row tiles per expert), then placement in
//                (t, r) order inside every expert
//   gemm gate/up A rows gathered by token index, B = dequantised gate rows and
//                up rows side by side; the epilogue applies SwiGLU and writes
//                H (fp16) in grouped order
//   gemm down    A = H, B = dequantised down rows -> Y (fp32) in grouped order
//   combine      y[t] = sum_r w[t][r] * Y[inv[t][r]], slot order fixed
//
// The grouped product (one CTA per 128 x 128 output tile, 160 threads):
// warps 0-3 each own one row of the A tile and one row of the B tile: they
// copy A with cp.async straight into the 128-byte swizzled K-major layout,
// copy the int8/int4 codes and scales of their B row, dequantise them to fp16
// (exact q*s rounded once) into the same layout, fence the writes for the
// async proxy and arrive on the stage's "full" barrier. One thread of warp 4
// issues tcgen05.mma (M=128, N=128, K=16, fp32 accumulator in TMEM) for each
// stage and commits to the stage's "empty" barrier; 4 stages of 64 along K are
// in flight. After the last stage warps 0-3 read the accumulator rows from
// TMEM (tcgen05.ld) and write the tile. Every wait is bounded.
#include <mutex>

#include "group.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace moe {

constexpr int kGM = 128;   // tile rows (tokens)
constexpr int kGN = 128;   // tile columns (B rows)
constexpr int kGK = 64;    // K per stage = one 128-byte row of 16-bit values
constexpr int kGS = 4;     // stages of A and B tiles
constexpr int kGThreads = 224;

// 8 codes (int8) -> 8 fp16 values q*s, rounded once.
__device__ __forceinline__ uint4 deq8_i8(uint2 w, float s) {
    uint32_t u0 = w.x ^ 0x80808080u, u1 = w.y ^ 0x80808080u;  // bias: byte = q + 128
    const __half2 magic = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    uint32_t p[4] = {__byte_perm(u0, 0x64646464u, 0x4140), __byte_perm(u0, 0x64646464u, 0x4342),
                     __byte_perm(u1, 0x64646464u, 0x4140), __byte_perm(u1, 0x64646464u, 0x4342)};
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        __half2 q = __hsub2(*reinterpret_cast<__half2*>(&p[i]), magic);  // exact q (|q| <= 128)
        float2 f = __half22float2(q);
        __half2 r = __floats2half2_rn(f.x * s, f.y * s);
        o[i] = *reinterpret_cast<uint32_t*>(&r);
    }
    return out;
}
// 8 codes (int4, one 32-bit word, element 2j in the low nibble of byte j).
__device__ __forceinline__ uint4 deq8_i4(uint32_t w, float s) {
    uint32_t u = w ^ 0x88888888u;  // nibble = q + 8
    const __half2 magic = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t v = u >> (8 * i);
        uint32_t p = (v & 0xFu) | ((v & 0xF0u) << 12) | 0x64006400u;
        __half2 q = __hsub2(*reinterpret_cast<__half2*>(&p), magic);
        float2 f = __half22float2(q);
        __half2 r = __floats2half2_rn(f.x * s, f.y * s);
        o[i] = *reinterpret_cast<uint32_t*>(&r);
    }
    return out;
}


template <int BMODE, typename ST>
struct GemmSmem {
    static constexpr int kR = BMODE == 16 ? 1 : (BMODE == 8 ? 8 : 12);  // raw code stages
    static constexpr int kRB = BMODE == 8 ? 64 : 32;                    // raw bytes per row per stage
    static constexpr int kAB = 2 * 16384;                               // A + B tile of one stage
    static constexpr int kRaw = BMODE == 16 ? 0 : kGN * kRB;
    static constexpr size_t kBytes = (size_t)kGS * kAB + (size_t)kR * kRaw + 1024;
};

// Warp roles (224 threads): warp 0 streams the int8/int4 codes of the B tile
// (TMA, kR stages ahead); warp 6 streams the A tile (TMA, 128-byte swizzle;
// also the B tile when B is already 16-bit); warps 1-4 dequantise one B row
// each into the swizzled layout and later run the epilogue; one thread of
// warp 5 issues the MMAs and owns the TMEM allocation.
template <int BMODE, typename ST, bool BF16, bool SWIGLU>
__global__ void __launch_bounds__(kGThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    using L = GemmSmem<BMODE, ST>;
    constexpr int R = L::kR;
    extern __shared__ unsigned char sm_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* ab = sm;                          // [kGS][A 16 KB | B 16 KB]
    unsigned char* raw = sm + (size_t)kGS * L::kAB;  // [R][128 rows][kRB]
    __shared__ __align__(8) uint64_t raw_full[R], raw_empty[R], a_full[kGS], b_full[kGS], ab_empty[kGS], done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x / p.n_ntiles, nt = blockIdx.x - (blockIdx.x / p.n_ntiles) * p.n_ntiles;
    pdl_wait();
    pdl_trigger();
    const int n_mt = p.n_mtiles_dev ? ld_cg_i32(p.n_mtiles_dev) : p.n_mtiles;
    if (mt >= n_mt) return;  // whole CTA, before any barrier or allocation
    const int g = p.tile_group ? ld_cg_i32(p.tile_group + mt) : 0;
    const int m0 = p.tile_m0 ? ld_cg_i32(p.tile_m0 + mt) : mt * kGM;
    const int m_end = p.group_end ? ld_cg_i32(p.group_end + g) : p.m_total;
    const int nk = p.K / kGK;
    int* status = &p.hdr->status;

    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < R; i++) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], 128);
        }
        for (int i = 0; i < kGS; i++) {
            mbar_init(&a_full[i], 1);
            mbar_init(&b_full[i], 128);
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
    const int brow0 = g * p.b_group_rows + nt * p.rows_per_ntile;  // B rows [0,64): brow0.. of map B0

    if (warp == 0) {
        // ------------------------------------------------ code producer
        if constexpr (BMODE != 16) {
            if (lane == 0) {
                for (int t = 0; t < nk; t++) {
                    const int s = t % R;
                    if (t >= R && !mbar_wait(&raw_empty[s], ((t / R) - 1) & 1, status)) {
                        s_abort = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&raw_full[s], kGN * L::kRB);
                    unsigned char* dst = raw + (size_t)s * L::kRaw;
                    tma_load_2d(dst, &p.tmB0, t * L::kRB, brow0, &raw_full[s]);
                    tma_load_2d(dst + 64 * L::kRB, &p.tmB1, t * L::kRB, brow0 + p.half_off, &raw_full[s]);
                }
            }
        }
    } else if (warp == 6) {
        // ------------------------------------------------ A producer
        if (lane == 0) {
            for (int t = 0; t < nk; t++) {
                const int s = t % kGS;
                if (t >= kGS && !mbar_wait(&ab_empty[s], ((t / kGS) - 1) & 1, status)) {
                    s_abort = 1;
                    break;
                }
                unsigned char* dst = ab + (size_t)s * L::kAB;
                mbar_arrive_expect_tx(&a_full[s], BMODE == 16 ? 32768 : 16384);
                tma_load_2d(dst, &p.tmA, t * kGK, m0, &a_full[s]);
                if constexpr (BMODE == 16) tma_load_2d(dst + 16384, &p.tmB0, t * kGK, brow0, &a_full[s]);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_f16(BF16, kGM, kGN);
            for (int t = 0; t < nk; t++) {
                const int s = t % kGS;
                const unsigned ph = (t / kGS) & 1;
                if (s_abort || !mbar_wait(&a_full[s], ph, status) ||
                    (BMODE != 16 && !mbar_wait(&b_full[s], ph, status))) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_addr(ab + (size_t)s * L::kAB);
                const uint64_t ad = umma_desc_sw128(a0), bd = umma_desc_sw128(a0 + 16384);
#pragma unroll
                for (int kk = 0; kk < kGK / 16; kk++)
                    umma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (t | kk) != 0 ? 1u : 0u);
                umma_commit(&ab_empty[s]);
            }
            umma_commit(&done);  // also after an abort: completes when the issued MMAs are done
        }
    } else {
        // ------------------------------------------------ dequant (warps 1-4)
        if constexpr (BMODE != 16) {
            const int j = tid - 32;  // B row of the tile
            const int half = j >> 6;
            const ST* Srow = reinterpret_cast<const ST*>(half ? p.S1 : p.S0) +
                             (size_t)(brow0 + (j & 63) + half * p.half_off) * (p.K / kBlk);
            float s0n = to_f32(Srow[0]), s1n = to_f32(Srow[1]);
            for (int t = 0; t < nk; t++) {
                const int rs = t % R, as = t % kGS;
                if (s_abort || !mbar_wait(&raw_full[rs], (t / R) & 1, status) ||
                    (t >= kGS && !mbar_wait(&ab_empty[as], ((t / kGS) - 1) & 1, status))) {
                    s_abort = 1;
                    break;
                }
                const float s0 = s0n, s1 = s1n;
                if (t + 1 < nk) {
                    s0n = to_f32(Srow[2 * t + 2]);
                    s1n = to_f32(Srow[2 * t + 3]);
                }
                const unsigned char* rr = raw + (size_t)rs * L::kRaw + j * L::kRB;
                unsigned char* bt = ab + (size_t)as * L::kAB + 16384;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    const float scl = c < 4 ? s0 : s1;
                    uint4 v;
                    if constexpr (BMODE == 8) v = deq8_i8(*reinterpret_cast<const uint2*>(rr + 8 * c), scl);
                    else v = deq8_i4(*reinterpret_cast<const uint32_t*>(rr + 4 * c), scl);
                    *reinterpret_cast<uint4*>(bt + sw128_off(j, c)) = v;
                }
                fence_proxy_async_smem();
                mbar_arrive(&raw_empty[rs]);
                mbar_arrive(&b_full[as]);
            }
        }
        // ------------------------------------------------ epilogue (warps 1-4)
        if (!mbar_wait(&done, 0, status)) s_abort = 1;
        tc_fence_after();
        const int row = 32 * (warp & 3) + lane;  // TMEM lane quarter of this warp
        const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const int pos = m0 + row;
        const bool valid = pos < m_end && !s_abort;
        if constexpr (SWIGLU) {
            __half* C = reinterpret_cast<__half*>(p.C) + (size_t)pos * p.ldc + nt * 64;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t gr[16], ur[16];
                tmem_ld16(trow + 16 * c, gr);
                tmem_ld16(trow + 64 + 16 * c, ur);
                tmem_ld_wait();
                uint32_t o[8];
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    float h0 = silu_mul(__uint_as_float(gr[2 * q]), __uint_as_float(ur[2 * q]));
                    float h1 = silu_mul(__uint_as_float(gr[2 * q + 1]), __uint_as_float(ur[2 * q + 1]));
                    __half2 hh = __floats2half2_rn(h0, h1);
                    o[q] = *reinterpret_cast<uint32_t*>(&hh);
                }
                if (valid) {
                    reinterpret_cast<uint4*>(C + 16 * c)[0] = make_uint4(o[0], o[1], o[2], o[3]);
                    reinterpret_cast<uint4*>(C + 16 * c)[1] = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
        } else {
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
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) tmem_dealloc(tmem, 128);
}

template <int BMODE, typename ST, bool BF16, bool SWIGLU>
static cudaError_t launch_gemm_t(const GemmParams& p, int max_mtiles, cudaStream_t s) {
    return launch(gemm_tc_kernel<BMODE, ST, BF16, SWIGLU>, dim3(max_mtiles * p.n_ntiles), dim3(kGThreads),
                  GemmSmem<BMODE, ST>::kBytes, s, true, p);
}

cudaError_t launch_gemm(const GemmParams& p, int bmode, bool s_f16, bool swiglu, int max_mtiles,
                        cudaStream_t s) {
    if (bmode == 16) return launch_gemm_t<16, float, true, false>(p, max_mtiles, s);
    if (bmode == 8) {
        if (swiglu) return s_f16 ? launch_gemm_t<8, __half, false, true>(p, max_mtiles, s)
                                 : launch_gemm_t<8, float, false, true>(p, max_mtiles, s);
        return s_f16 ? launch_gemm_t<8, __half, false, false>(p, max_mtiles, s)
                     : launch_gemm_t<8, float, false, false>(p, max_mtiles, s);
    }
    if (swiglu) return s_f16 ? launch_gemm_t<4, __half, false, true>(p, max_mtiles, s)
                             : launch_gemm_t<4, float, false, true>(p, max_mtiles, s);
    return s_f16 ? launch_gemm_t<4, __half, false, false>(p, max_mtiles, s)
                 : launch_gemm_t<4, float, false, false>(p, max_mtiles, s);
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

bool make_tmap_2d(CUtensorMap* m, int dtype, const void* base, unsigned long long inner, unsigned long long rows,
                  unsigned long long row_bytes, unsigned box_inner, unsigned box_rows, int swizzle) {
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
