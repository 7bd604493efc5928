// Grouped expert projections of the prefill on the 5th-generation tensor
// cores, weights stationary.
//
// Qiita "custom Metal gather_qmm" (sections 4 and 7): the gate and up
// projections share each token's x, SwiGLU joins them, down maps the
// activation back, and only routed experts' weights are read. With many tokens
// per expert these are dense contractions, one per (expert, projection).
//
// Work item = (tile of up to NT consecutive grouped positions of one expert,
// block of 128 weight rows). The weight block is the MMA's A operand (M = 128):
// its int8/int4 codes arrive by TMA and are dequantised to fp16 in shared
// memory once per K stage; the tokens' 16-bit rows are the B operand
// (N = the tile's token count rounded up to 16, at most NT), also by TMA; the
// fp32 accumulator D[weight row][token] lives in tensor memory, two buffers of
// NT columns, so that the epilogue of one item overlaps the MMAs of the next.
// The grid is persistent: CTA c takes items c, c + G, ...; consecutive items
// share their token tile (read from L2) and cover the expert's weight blocks.
//
// Gate/up (SwiGLU): A row 2i is gate row f0 + i and row 2i + 1 is up row
// f0 + i, so a unit's two accumulators sit in neighbouring TMEM lanes of one
// warp and the epilogue pairs them with one shuffle; it writes
// H[pos][f] = silu(g) * u in fp16. Down: A row j is down row d0 + j and the
// epilogue writes Y[pos][d] in fp32.
//
// Warp roles (15 warps): 0 code producer (TMA, R stages ahead; the code tiles
// are swizzled across their 64- or 32-byte rows so that the dequantising
// reads hit all banks), 1 token producer (TMA) and TMEM owner, 2 MMA issuer,
// 3-10 dequantisation (two threads per A row, each one 32-code scale block of
// the stage), 11-14 epilogue (TMEM lane quarter = warp % 4). Every wait is
// bounded; a timeout records MOE_ERR_DEVICE_TIMEOUT and ends the CTA's loops.
#include "kernels.h"
#include "tc.cuh"

namespace moe {

constexpr int kEK = 64;          // K per stage: one 128-byte row of 16-bit values
constexpr int kEThreads = 480;   // 15 warps
constexpr int kEDeq = 256;       // dequantising threads

template <int QB, int NT>
struct EgSmem {
    static constexpr int kRB = QB == 8 ? 64 : 32;        // code bytes per row per stage
    static constexpr int kRaw = 128 * kRB;               // one code stage
    static constexpr int kS = NT == 256 ? 3 : 4;         // A/B stages
    static constexpr int kR = NT == 256 ? (QB == 8 ? 8 : 12) : (QB == 8 ? 10 : 16);  // code stages
    static constexpr int kA = 128 * 128;                 // 128 rows x 64 fp16
    static constexpr int kB = NT * 128;                  // NT rows x 64 fp16
    static constexpr size_t kBytes = (size_t)kS * (kA + kB) + (size_t)kR * kRaw + 1024;
};

// 8 int8 codes -> 8 fp16 values q*s (exact q, one rounding of the product).
__device__ __forceinline__ uint4 deq8_i8(uint2 w, __half2 s2) {
    const uint32_t u0 = w.x ^ 0x80808080u, u1 = w.y ^ 0x80808080u;  // byte = q + 128
    const __half2 magic = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    const uint32_t pk[4] = {__byte_perm(u0, 0x64646464u, 0x4140), __byte_perm(u0, 0x64646464u, 0x4342),
                            __byte_perm(u1, 0x64646464u, 0x4140), __byte_perm(u1, 0x64646464u, 0x4342)};
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&pk[i]), magic);  // 1024 + b - 1152
        const __half2 r = __hmul2(q, s2);
        o[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
    return out;
}
__device__ __forceinline__ uint4 deq8_i8(uint2 w, float s) {
    const uint32_t u0 = w.x ^ 0x80808080u, u1 = w.y ^ 0x80808080u;
    const __half2 magic = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const uint32_t pk[4] = {__byte_perm(u0, 0x64646464u, 0x4140), __byte_perm(u0, 0x64646464u, 0x4342),
                            __byte_perm(u1, 0x64646464u, 0x4140), __byte_perm(u1, 0x64646464u, 0x4342)};
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 f = __half22float2(__hsub2(*reinterpret_cast<const __half2*>(&pk[i]), magic));
        const __half2 r = __floats2half2_rn(f.x * s, f.y * s);
        o[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
    return out;
}
// 8 int4 codes (one word, element 2j in the low nibble of byte j).
__device__ __forceinline__ uint4 deq8_i4(uint32_t w, __half2 s2) {
    const uint32_t u = w ^ 0x88888888u;  // nibble = q + 8
    const __half2 magic = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint32_t v = u >> (8 * i);
        const uint32_t pk = (v & 0xFu) | ((v & 0xF0u) << 12) | 0x64006400u;
        const __half2 r = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&pk), magic), s2);
        o[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
    return out;
}
__device__ __forceinline__ uint4 deq8_i4(uint32_t w, float s) {
    const uint32_t u = w ^ 0x88888888u;
    const __half2 magic = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint32_t v = u >> (8 * i);
        const uint32_t pk = (v & 0xFu) | ((v & 0xF0u) << 12) | 0x64006400u;
        const float2 f = __half22float2(__hsub2(*reinterpret_cast<const __half2*>(&pk), magic));
        const __half2 r = __floats2half2_rn(f.x * s, f.y * s);
        o[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
    return out;
}

// One work item, as every role decodes it.
struct EgItem {
    int e, wb, m0, n;  // expert, weight block, first position, positions (1..NT)
};
template <int NT>
__device__ __forceinline__ EgItem eg_item(const EgParams& p, int i) {
    EgItem it;
    const int ti = i / p.nwb;
    it.wb = i - ti * p.nwb;
    it.e = ld_cg_i32(p.tile_group + ti);
    it.m0 = ld_cg_i32(p.tile_m0 + ti);
    const int end = ld_cg_i32(p.group_end + it.e);
    it.n = min(NT, end - it.m0);
    return it;
}

template <int QB, typename ST, int NT, bool SWIGLU>
__global__ void __launch_bounds__(kEThreads, 1) egemm_kernel(const __grid_constant__ EgParams p) {
    using L = EgSmem<QB, NT>;
    constexpr int R = L::kR, S = L::kS;
    extern __shared__ unsigned char sm_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* sa = sm;                                   // [S][A 16 KB]
    unsigned char* sb = sm + (size_t)S * L::kA;               // [S][B NT*128 B]
    unsigned char* raw = sb + (size_t)S * L::kB;              // [R][128 rows][kRB]
    __shared__ __align__(8) uint64_t raw_full[R], raw_empty[R], a_full[S], b_full[S], ab_empty[S];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* status = &p.hdr->status;
    const int nk = p.K / kEK;
    const int G = gridDim.x;

    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < R; i++) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kEDeq);
        }
        for (int i = 0; i < S; i++) {
            mbar_init(&a_full[i], kEDeq);
            mbar_init(&b_full[i], 1);
            mbar_init(&ab_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 128);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&s_tmem, 2 * NT);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    pdl_wait();
    pdl_trigger();
    const int n_items = ld_cg_i32(p.n_tiles_dev) * p.nwb;

    if (warp == 0) {
        // ------------------------------------------------ code producer
        if (lane == 0) {
            int kt = 0;
            for (int i = blockIdx.x; i < n_items && !s_abort; i += G) {
                const EgItem it = eg_item<NT>(p, i);
                const int row0 = it.e * p.w_rows + it.wb * (SWIGLU ? 64 : 128);
                const int row1 = SWIGLU ? row0 : row0 + 64;
                for (int t = 0; t < nk; t++, kt++) {
                    const int s = kt % R;
                    if (kt >= R && !mbar_wait(&raw_empty[s], ((kt / R) - 1) & 1, status)) {
                        s_abort = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&raw_full[s], L::kRaw);
                    unsigned char* dst = raw + (size_t)s * L::kRaw;
                    tma_load_2d(dst, &p.tmW0, t * L::kRB, row0, &raw_full[s]);
                    tma_load_2d(dst + 64 * L::kRB, &p.tmW1, t * L::kRB, row1, &raw_full[s]);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ token producer
        if (lane == 0) {
            int kt = 0;
            for (int i = blockIdx.x; i < n_items && !s_abort; i += G) {
                const EgItem it = eg_item<NT>(p, i);
                for (int t = 0; t < nk; t++, kt++) {
                    const int s = kt % S;
                    if (kt >= S && !mbar_wait(&ab_empty[s], ((kt / S) - 1) & 1, status)) {
                        s_abort = 1;
                        break;
                    }
                    const bool half = it.n <= NT / 2;  // the MMA reads only N <= NT/2 rows then
                    mbar_arrive_expect_tx(&b_full[s], half ? L::kB / 2 : L::kB);
                    tma_load_2d(sb + (size_t)s * L::kB, half ? &p.tmXh : &p.tmX, t * kEK, it.m0, &b_full[s]);
                }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int kt = 0, li = 0;
            for (int i = blockIdx.x; i < n_items && !s_abort; i += G, li++) {
                const EgItem it = eg_item<NT>(p, i);
                const int buf = li & 1;
                if (li >= 2 && !mbar_wait(&acc_empty[buf], ((li >> 1) - 1) & 1, status)) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const int N = (it.n + 15) & ~15;
                const uint32_t idesc = umma_idesc_f16(false, 128, N);
                const uint32_t d = tmem + (uint32_t)(buf * NT);
                for (int t = 0; t < nk; t++, kt++) {
                    const int s = kt % S;
                    const unsigned ph = (kt / S) & 1;
                    if (s_abort || !mbar_wait(&a_full[s], ph, status) || !mbar_wait(&b_full[s], ph, status)) {
                        s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = umma_desc_sw128(smem_addr(sa + (size_t)s * L::kA));
                    const uint64_t bd = umma_desc_sw128(smem_addr(sb + (size_t)s * L::kB));
#pragma unroll
                    for (int kk = 0; kk < kEK / 16; kk++)
                        umma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, (t | kk) != 0 ? 1u : 0u);
                    umma_commit(&ab_empty[s]);
                }
                umma_commit(&acc_full[buf]);  // also after an abort: completes when the issued MMAs are done
            }
        }
    } else if (warp >= 3 && warp <= 10) {
        // ------------------------------------------------ dequantisation
        const int j = tid - 96;                                   // 0 .. 255
        const int row = j >> 1, h = j & 1;                        // A row; 32-code half of the stage
        const int rr = SWIGLU ? ((row & 1) * 64 + (row >> 1)) : row;  // its code row in a stage
        // 16-byte chunk c of code row r sits at chunk c ^ swz(r) (TMA swizzle)
        const int swz = QB == 8 ? ((rr >> 1) & 3) : ((rr >> 2) & 1);
        const int nsb = p.K / kBlk;                               // scales per weight row
        constexpr int SPV = 16 / (int)sizeof(ST);                 // scales per 16-byte vector
        constexpr int TPV = SPV / 2;                              // stages per vector
        const bool vec = (nsb * (int)sizeof(ST)) % 16 == 0;
        int kt = 0;
        for (int i = blockIdx.x; i < n_items && !s_abort; i += G) {
            const EgItem it = eg_item<NT>(p, i);
            const int wrow = it.e * p.w_rows + (SWIGLU ? it.wb * 64 + (row >> 1) : it.wb * 128 + row);
            const ST* srow = reinterpret_cast<const ST*>(SWIGLU && (row & 1) ? p.S1 : p.S0) + (size_t)wrow * nsb;
            // this thread's scale (block 2t + h) per stage: from 16-byte vectors
            // loaded two ahead, or one value loaded one stage ahead
            uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0, v2 = v0;
            const int nvec = (nsb + SPV - 1) / SPV;
            float snext = 0.f;
            if (vec) {
                v0 = ld_nc16(srow);
                if (nvec > 1) v1 = ld_nc16(srow + SPV);
                if (nvec > 2) v2 = ld_nc16(srow + 2 * SPV);
            } else {
                snext = to_f32(srow[h]);
            }
            for (int t = 0; t < nk; t++, kt++) {
                const int rs = kt % R, as = kt % S;
                if (s_abort || !mbar_wait(&raw_full[rs], (kt / R) & 1, status) ||
                    (kt >= S && !mbar_wait(&ab_empty[as], ((kt / S) - 1) & 1, status))) {
                    s_abort = 1;
                    break;
                }
                float sc;
                if (vec) {
                    if (t > 0 && t % TPV == 0) {
                        v0 = v1;
                        v1 = v2;
                        const int vn = t / TPV + 2;
                        if (vn < nvec) v2 = ld_nc16(srow + vn * SPV);
                    }
                    const int q = t % TPV;
                    if constexpr (sizeof(ST) == 2) {
                        const uint32_t w2 = q == 0 ? v0.x : q == 1 ? v0.y : q == 2 ? v0.z : v0.w;
                        sc = __half2float(__ushort_as_half((unsigned short)(h ? (w2 >> 16) : (w2 & 0xFFFFu))));
                    } else {
                        const uint32_t w2 = q == 0 ? (h ? v0.y : v0.x) : (h ? v0.w : v0.z);
                        sc = __uint_as_float(w2);
                    }
                } else {
                    sc = snext;
                    if (t + 1 < nk) snext = to_f32(srow[2 * t + 2 + h]);
                }
                const unsigned char* rp = raw + (size_t)rs * L::kRaw + rr * L::kRB;
                unsigned char* at = sa + (size_t)as * L::kA;
                uint4 c0, c1;
                if constexpr (QB == 8) {
                    c0 = *reinterpret_cast<const uint4*>(rp + 16 * ((2 * h) ^ swz));
                    c1 = *reinterpret_cast<const uint4*>(rp + 16 * ((2 * h + 1) ^ swz));
                } else {
                    c0 = *reinterpret_cast<const uint4*>(rp + 16 * (h ^ swz));
                }
                uint4 o[4];
                if constexpr (sizeof(ST) == 2) {
                    const __half2 s2 = __float2half2_rn(sc);  // exact: sc is an fp16 value
                    if constexpr (QB == 8) {
                        o[0] = deq8_i8(make_uint2(c0.x, c0.y), s2);
                        o[1] = deq8_i8(make_uint2(c0.z, c0.w), s2);
                        o[2] = deq8_i8(make_uint2(c1.x, c1.y), s2);
                        o[3] = deq8_i8(make_uint2(c1.z, c1.w), s2);
                    } else {
                        o[0] = deq8_i4(c0.x, s2);
                        o[1] = deq8_i4(c0.y, s2);
                        o[2] = deq8_i4(c0.z, s2);
                        o[3] = deq8_i4(c0.w, s2);
                    }
                } else {
                    if constexpr (QB == 8) {
                        o[0] = deq8_i8(make_uint2(c0.x, c0.y), sc);
                        o[1] = deq8_i8(make_uint2(c0.z, c0.w), sc);
                        o[2] = deq8_i8(make_uint2(c1.x, c1.y), sc);
                        o[3] = deq8_i8(make_uint2(c1.z, c1.w), sc);
                    } else {
                        o[0] = deq8_i4(c0.x, sc);
                        o[1] = deq8_i4(c0.y, sc);
                        o[2] = deq8_i4(c0.z, sc);
                        o[3] = deq8_i4(c0.w, sc);
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; c++) *reinterpret_cast<uint4*>(at + sw128_off(row, 4 * h + c)) = o[c];
                fence_proxy_async_smem();
                mbar_arrive(&raw_empty[rs]);
                mbar_arrive(&a_full[as]);
            }
        }
    } else if (warp >= 11) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quarter
        const int j = 32 * q + lane;          // A row = TMEM lane
        int li = 0;
        for (int i = blockIdx.x; i < n_items && !s_abort; i += G, li++) {
            const EgItem it = eg_item<NT>(p, i);
            const int buf = li & 1;
            if (!mbar_wait(&acc_full[buf], (li >> 1) & 1, status)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * NT);
            const int N = (it.n + 15) & ~15;
            for (int c0 = 0; c0 < N; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tb + c0, v);
                tmem_ld_wait();
                if constexpr (SWIGLU) {
                    // even lane: gate of unit f, columns c0..c0+7; odd lane: up
                    // of unit f, columns c0+8..c0+15 (each gets the other half)
                    const bool odd = lane & 1;
                    const int f = it.wb * 64 + (j >> 1);
                    __half* H = reinterpret_cast<__half*>(p.C);
#pragma unroll
                    for (int i2 = 0; i2 < 8; i2++) {
                        const uint32_t mine = odd ? v[i2] : v[8 + i2];
                        const uint32_t other = __shfl_xor_sync(kFull, mine, 1);
                        const float g = __uint_as_float(odd ? other : v[i2]);
                        const float u = __uint_as_float(odd ? v[8 + i2] : other);
                        const int col = c0 + (odd ? 8 : 0) + i2;
                        if (col < it.n) H[(size_t)(it.m0 + col) * p.ldc + f] = __float2half_rn(silu_mul(g, u));
                    }
                } else {
                    float* Y = reinterpret_cast<float*>(p.C);
                    const int dcol = it.wb * 128 + j;
#pragma unroll
                    for (int i2 = 0; i2 < 16; i2++) {
                        const int col = c0 + i2;
                        if (col < it.n) Y[(size_t)(it.m0 + col) * p.ldc + dcol] = __uint_as_float(v[i2]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * NT);
}

template <int QB, typename ST, int NT, bool SWIGLU>
static cudaError_t launch_egemm_t(const EgParams& p, int grid, cudaStream_t s) {
    return launch(egemm_kernel<QB, ST, NT, SWIGLU>, dim3(grid), dim3(kEThreads), EgSmem<QB, NT>::kBytes, s, true, p);
}

template <int NT>
static cudaError_t launch_egemm_nt(const EgParams& p, int qbits, bool s_f16, bool swiglu, int grid, cudaStream_t s) {
    if (qbits == 8) {
        if (swiglu) return s_f16 ? launch_egemm_t<8, __half, NT, true>(p, grid, s)
                                 : launch_egemm_t<8, float, NT, true>(p, grid, s);
        return s_f16 ? launch_egemm_t<8, __half, NT, false>(p, grid, s)
                     : launch_egemm_t<8, float, NT, false>(p, grid, s);
    }
    if (swiglu) return s_f16 ? launch_egemm_t<4, __half, NT, true>(p, grid, s)
                             : launch_egemm_t<4, float, NT, true>(p, grid, s);
    return s_f16 ? launch_egemm_t<4, __half, NT, false>(p, grid, s)
                 : launch_egemm_t<4, float, NT, false>(p, grid, s);
}

cudaError_t launch_egemm(const EgParams& p, int qbits, bool s_f16, bool swiglu, int nt, int grid, cudaStream_t s) {
    return nt == 256 ? launch_egemm_nt<256>(p, qbits, s_f16, swiglu, grid, s)
                     : launch_egemm_nt<128>(p, qbits, s_f16, swiglu, grid, s);
}

}  // namespace moe
