// Grouped expert projections on the 5th-generation tensor cores, weights
// stationary: the prefill, and decode of four or more tokens.
//
// Qiita "custom Metal gather_qmm" (sections 4 and 7): the gate and up
// projections share each token's x, SwiGLU joins them, down maps the
// activation back, and only routed experts' weights are read. With many tokens
// per expert these are dense contractions, one per (expert, projection).
//
// Work item = (tile of up to 128 consecutive grouped positions of one expert,
// block of 128 weight rows). The weight block is the MMA's A operand (M = 128):
// its int8/int4 codes arrive by TMA, are dequantised to fp16 in registers and
// written to TENSOR MEMORY (tcgen05.st), from where the MMA reads them; the
// tokens' 16-bit rows are the B operand (N = the tile's token count rounded up
// to 16), from shared memory by TMA. With A in tensor memory a K stage moves
// only the code tile and the token tile through shared memory (32-48 KB
// instead of 64-80 KB with A staged there as well).
// Tensor memory (512 columns): two fp32 accumulators of 128 columns, so that
// the epilogue of one item overlaps the MMAs of the next, and a ring of 6 A
// stages of 32 columns (128 rows x 64 fp16). Each tcgen05 instruction costs
// the single issuing thread tens of cycles, so the issuer commits once per
// pair of stages (freeing both stages' A and B slots).
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
// 3-10 dequantisation (TMEM lane quarter = warp % 4, one A row per thread;
// warps 3-6 take the even stages, 7-10 the odd ones), 11-14 epilogue (lane
// quarter = warp % 4). Every wait is bounded; a timeout records
// MOE_ERR_DEVICE_TIMEOUT and ends the CTA's loops.
#include <type_traits>

#include "kernels.h"
#include "tc.cuh"

namespace moe {

constexpr int kEK = 64;          // K per stage: 64 16-bit values = 32 TMEM columns
constexpr int kENT = 128;        // token tile (MMA N at most)
constexpr int kEThreads = 480;   // 15 warps
constexpr int kEDeq = 256;       // dequantising threads
constexpr int kES = 6;           // A stages (tensor memory) = B stages (shared memory); even
constexpr uint32_t kEAcc = 2 * kENT;  // first TMEM column of the A stages

template <int QB>
struct EgSmem {
    static constexpr int kRB = QB == 8 ? 64 : 32;        // code bytes per row per stage
    static constexpr int kRaw = 128 * kRB;               // one code stage
    static constexpr int kSB = kES;                      // token (B) stages
    static constexpr int kR = QB == 8 ? 12 : 20;         // code stages
    static constexpr int kB = kENT * 128;                // 128 rows x 64 fp16
    static constexpr size_t kBytes = (size_t)kSB * kB + (size_t)kR * kRaw + 1024;
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
__device__ __forceinline__ EgItem eg_item_load(const EgParams& p, int i) {
    EgItem it;
    const int ti = i / p.nwb;
    it.wb = i - ti * p.nwb;
    it.e = ld_cg_i32(p.tile_group + ti);
    it.m0 = ld_cg_i32(p.tile_m0 + ti);
    it.n = ld_cg_i32(p.tile_n + ti);
    return it;
}
constexpr int kEgItems = 256;  // items of one CTA kept in shared memory

template <int QB, typename ST, bool SWIGLU>
__global__ void __launch_bounds__(kEThreads, 1) egemm_kernel(const __grid_constant__ EgParams p) {
    using L = EgSmem<QB>;
    constexpr int R = L::kR, S = kES, NT = kENT;
    extern __shared__ unsigned char sm_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* sb = sm;                                   // [S][B 16 KB]
    unsigned char* raw = sb + (size_t)S * L::kB;              // [R][128 rows][kRB]
    // ab_empty[s/2]: both A and B slots of stages s and s+1 (s even) free again;
    // the MMA issuer commits once per pair of stages
    __shared__ __align__(8) uint64_t raw_full[R], raw_empty[R], a_full[S], b_full[S], ab_empty[S / 2];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ EgItem s_items[kEgItems];
    __shared__ int s_pexp[2][kENT];  // scale exponents of the item's positions, per accumulator buffer

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* status = &p.hdr->status;
    const int nk = p.K / kEK;
    const int G = gridDim.x;

    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < R; i++) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kEDeq / 2);  // one group of dequantising warps per stage
        }
        for (int i = 0; i < S; i++) {
            mbar_init(&a_full[i], kEDeq / 2);
            mbar_init(&b_full[i], 1);
        }
        for (int i = 0; i < S / 2; i++) mbar_init(&ab_empty[i], 1);
        for (int i = 0; i < 2; i++) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 128);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    pdl_wait();
    pdl_trigger();
    const int n_items = ld_cg_i32(p.n_tiles_dev) * p.nwb;
    // this CTA's items c, c + G, ... : the first kEgItems decoded once into
    // shared memory (all loads in flight together), later ones on the fly
    if (warp == 3)
        for (int li = lane; li < kEgItems; li += 32) {
            const int i = blockIdx.x + li * G;
            if (i < n_items) s_items[li] = eg_item_load(p, i);
        }
    __syncthreads();
    auto eg_item = [&](int i) -> EgItem {
        const int li = (i - (int)blockIdx.x) / G;
        return li < kEgItems ? s_items[li] : eg_item_load(p, i);
    };

    if (warp == 0) {
        // ------------------------------------------------ code producer
        if (lane == 0) {
            int kt = 0;
            for (int i = blockIdx.x; i < n_items && !s_abort; i += G) {
                const EgItem it = eg_item(i);
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
                const EgItem it = eg_item(i);
                const bool half = it.n <= NT / 2;  // the MMA reads only N <= NT/2 rows then
                for (int t = 0; t < nk; t++, kt++) {
                    const int s = kt % S;
                    if (kt >= S && !mbar_wait(&ab_empty[s >> 1], ((kt / S) - 1) & 1, status)) {
                        s_abort = 1;
                        break;
                    }
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
                const EgItem it = eg_item(i);
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
                    if (s_abort || !mbar_wait(&a_full[s], (kt / S) & 1, status) ||
                        !mbar_wait(&b_full[s], (kt / S) & 1, status)) {
                        s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t at = tmem + kEAcc + (uint32_t)(32 * s);
                    const uint64_t bd = umma_desc_sw128(smem_addr(sb + (size_t)s * L::kB));
#pragma unroll
                    for (int kk = 0; kk < kEK / 16; kk++)
                        umma_f16_ts(d, at + 8 * kk, bd + 2 * kk, idesc, (t | kk) != 0 ? 1u : 0u);
                    if (s & 1) umma_commit(&ab_empty[s >> 1]);  // frees stages s-1 and s
                }
                umma_commit(&acc_full[buf]);  // also after an abort: completes when the issued MMAs are done
            }
        }
    } else if (warp >= 3 && warp <= 10) {
        // ------------------------------------------------ dequantisation
        // two groups of four warps take alternate stages, so that one stage's
        // latency (waits, loads, conversion, TMEM store) overlaps the other's
        const int q = warp & 3;                                   // TMEM lane quarter
        const int row = 32 * q + lane;                            // A row = TMEM lane
        const int grp = (warp - 3) >> 2;                          // stages kt with kt % 2 == grp
        const int rr = SWIGLU ? ((row & 1) * 64 + (row >> 1)) : row;  // its code row in a stage
        // 16-byte chunk c of code row r sits at chunk c ^ swz(r) (TMA swizzle)
        const int swz = QB == 8 ? ((rr >> 1) & 3) : ((rr >> 2) & 1);
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + kEAcc;
        const int nsb = p.K / kBlk;                               // scales per weight row (2 per stage)
        int kt = 0;
        for (int i = blockIdx.x; i < n_items && !s_abort; i += G) {
            const EgItem it = eg_item(i);
            const int wrow = it.e * p.w_rows + (SWIGLU ? it.wb * 64 + (row >> 1) : it.wb * 128 + row);
            const ST* srow = reinterpret_cast<const ST*>(SWIGLU && (row & 1) ? p.S1 : p.S0) + (size_t)wrow * nsb;
            // the two scales of stage t as one 4-byte (fp16) or 8-byte (fp32) load
            using SP = typename std::conditional<sizeof(ST) == 2, uint32_t, uint2>::type;
            auto ld_sp = [&](int t) -> SP { return __ldg(reinterpret_cast<const SP*>(srow + 2 * t)); };
            // this group's first two stages of the item, loaded ahead
            int t0 = ((kt & 1) == grp) ? 0 : 1;
            SP sq0 = {}, sq1 = {};
            if (t0 < nk) sq0 = ld_sp(t0);
            if (t0 + 2 < nk) sq1 = ld_sp(t0 + 2);
            for (int t = 0; t < nk; t++, kt++) {
                if ((kt & 1) != grp) continue;
                const int rs = kt % R, as = kt % S;
                if (s_abort || !mbar_wait(&raw_full[rs], (kt / R) & 1, status) ||
                    (kt >= S && !mbar_wait(&ab_empty[as >> 1], ((kt / S) - 1) & 1, status))) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const SP sp = sq0;
                sq0 = sq1;
                if (t + 4 < nk) sq1 = ld_sp(t + 4);
                float s0, s1;
                if constexpr (sizeof(ST) == 2) {
                    s0 = __half2float(__ushort_as_half((unsigned short)(sp & 0xFFFFu)));
                    s1 = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
                } else {
                    s0 = __uint_as_float(sp.x);
                    s1 = __uint_as_float(sp.y);
                }
                const unsigned char* rp = raw + (size_t)rs * L::kRaw + rr * L::kRB;
                uint32_t cols[32];
                if constexpr (QB == 8) {
                    uint4 c[4];
#pragma unroll
                    for (int cc = 0; cc < 4; cc++) c[cc] = *reinterpret_cast<const uint4*>(rp + 16 * (cc ^ swz));
                    mbar_arrive(&raw_empty[rs]);  // the code tile is read
#pragma unroll
                    for (int cc = 0; cc < 4; cc++) {
                        uint4 o0, o1;
                        if constexpr (sizeof(ST) == 2) {
                            const __half2 s2 = __float2half2_rn(cc < 2 ? s0 : s1);  // exact: fp16 values
                            o0 = deq8_i8(make_uint2(c[cc].x, c[cc].y), s2);
                            o1 = deq8_i8(make_uint2(c[cc].z, c[cc].w), s2);
                        } else {
                            o0 = deq8_i8(make_uint2(c[cc].x, c[cc].y), cc < 2 ? s0 : s1);
                            o1 = deq8_i8(make_uint2(c[cc].z, c[cc].w), cc < 2 ? s0 : s1);
                        }
                        cols[8 * cc] = o0.x; cols[8 * cc + 1] = o0.y; cols[8 * cc + 2] = o0.z; cols[8 * cc + 3] = o0.w;
                        cols[8 * cc + 4] = o1.x; cols[8 * cc + 5] = o1.y; cols[8 * cc + 6] = o1.z; cols[8 * cc + 7] = o1.w;
                    }
                } else {
                    uint4 c[2];
#pragma unroll
                    for (int cc = 0; cc < 2; cc++) c[cc] = *reinterpret_cast<const uint4*>(rp + 16 * (cc ^ swz));
                    mbar_arrive(&raw_empty[rs]);
#pragma unroll
                    for (int cc = 0; cc < 2; cc++) {
                        const uint32_t w4[4] = {c[cc].x, c[cc].y, c[cc].z, c[cc].w};
#pragma unroll
                        for (int wq = 0; wq < 4; wq++) {
                            uint4 o;
                            if constexpr (sizeof(ST) == 2) o = deq8_i4(w4[wq], __float2half2_rn(cc ? s1 : s0));
                            else o = deq8_i4(w4[wq], cc ? s1 : s0);
                            cols[16 * cc + 4 * wq] = o.x; cols[16 * cc + 4 * wq + 1] = o.y;
                            cols[16 * cc + 4 * wq + 2] = o.z; cols[16 * cc + 4 * wq + 3] = o.w;
                        }
                    }
                }
                uint32_t lo[16], hi[16];
#pragma unroll
                for (int c2 = 0; c2 < 16; c2++) {
                    lo[c2] = cols[c2];
                    hi[c2] = cols[16 + c2];
                }
                tmem_st16(tq + (uint32_t)(32 * as), lo);
                tmem_st16(tq + (uint32_t)(32 * as + 16), hi);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&a_full[as]);
            }
        }
    } else if (warp >= 11) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quarter
        const int j = 32 * q + lane;          // A row = TMEM lane
        int li = 0;
        for (int i = blockIdx.x; i < n_items && !s_abort; i += G, li++) {
            const EgItem it = eg_item(i);
            const int buf = li & 1;
            if (!mbar_wait(&acc_full[buf], (li >> 1) & 1, status)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * NT);
            const int N = (it.n + 15) & ~15;
            // the item's position exponents, once, into shared memory (the four
            // epilogue warps meet on named barrier 1)
            s_pexp[buf][j] = j < it.n ? ld_cg_i32(p.pexp + it.m0 + j) : 0;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            // 2^k as an exact fp32 factor (|k| <= 120, split in two steps)
            auto pow2 = [](int kk) {
                const int a = kk / 2;
                return __int_as_float((127 + a) << 23) * __int_as_float((127 + kk - a) << 23);
            };
            for (int c0 = 0; c0 < N; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tb + c0, v);
                tmem_ld_wait();
                if constexpr (SWIGLU) {
                    // even lane: gate of unit f, columns c0..c0+7; odd lane: up
                    // of unit f, columns c0+8..c0+15 (each gets the other half).
                    // The accumulators are x*2^-e products: g, u = acc * 2^e; h
                    // is stored as h * 2^-2e (the down product undoes it).
                    const bool odd = lane & 1;
                    const int f = it.wb * 64 + (j >> 1);
                    __half* H = reinterpret_cast<__half*>(p.C);
#pragma unroll
                    for (int i2 = 0; i2 < 8; i2++) {
                        const uint32_t mine = odd ? v[i2] : v[8 + i2];
                        const uint32_t other = __shfl_xor_sync(kFull, mine, 1);
                        const int col = c0 + (odd ? 8 : 0) + i2;
                        const int ex = s_pexp[buf][col];
                        const float up = pow2(ex);
                        const float g = __uint_as_float(odd ? other : v[i2]) * up;
                        const float u = __uint_as_float(odd ? v[8 + i2] : other) * up;
                        if (col < it.n)
                            H[(size_t)(it.m0 + col) * p.ldc + f] = __float2half_rn(silu_mul(g, u) * pow2(-2 * ex));
                    }
                } else {
                    float* Y = reinterpret_cast<float*>(p.C);
                    const int dcol = it.wb * 128 + j;
#pragma unroll
                    for (int i2 = 0; i2 < 16; i2++) {
                        const int col = c0 + i2;
                        if (col < it.n) {
                            const int ex = s_pexp[buf][col];
                            Y[(size_t)(it.m0 + col) * p.ldc + dcol] = __uint_as_float(v[i2]) * pow2(2 * ex);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int QB, typename ST, bool SWIGLU>
static cudaError_t launch_egemm_t(const EgParams& p, int grid, cudaStream_t s) {
    return launch(egemm_kernel<QB, ST, SWIGLU>, dim3(grid), dim3(kEThreads), EgSmem<QB>::kBytes, s, true, p);
}

cudaError_t launch_egemm(const EgParams& p, int qbits, bool s_f16, bool swiglu, int grid, cudaStream_t s) {
    if (qbits == 8) {
        if (swiglu) return s_f16 ? launch_egemm_t<8, __half, true>(p, grid, s) : launch_egemm_t<8, float, true>(p, grid, s);
        return s_f16 ? launch_egemm_t<8, __half, false>(p, grid, s) : launch_egemm_t<8, float, false>(p, grid, s);
    }
    if (swiglu) return s_f16 ? launch_egemm_t<4, __half, true>(p, grid, s) : launch_egemm_t<4, float, true>(p, grid, s);
    return s_f16 ? launch_egemm_t<4, __half, false>(p, grid, s) : launch_egemm_t<4, float, false>(p, grid, s);
}

}  // namespace moe
