// Test scaffolding: lets csrc/edge0.cu compile as plain C++ on the CPU, in
// place of the library's kernels.h. It supplies the few CUDA builtins and
// library helpers that file uses. A launch runs the blocks and their warps one
// after another; the 32 lanes of a warp are fibers (ucontext) on one thread,
// which meet at every shuffle, so a warp reduction runs in lockstep as on the
// GPU. Valid only for kernels without shared memory or block barriers (those
// of edge0.cu). A 16-byte load of an unaligned address aborts, as the GPU
// would fault.
#pragma once
#include <algorithm>
#include <atomic>
#include <ucontext.h>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>

#include "moe_route.h"

#define __global__
#define __device__
#define __forceinline__ inline
#define __launch_bounds__(x)

struct dim3 {
    unsigned x, y, z;
    dim3(unsigned a = 1, unsigned b = 1, unsigned c = 1) : x(a), y(b), z(c) {}
};
struct uint4 { uint32_t x, y, z, w; };
inline uint4 make_uint4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) { return {a, b, c, d}; }
typedef int cudaError_t;
constexpr int cudaSuccess = 0;
typedef void* cudaStream_t;
struct __half { uint16_t b; };
struct __nv_bfloat16 { uint16_t b; };

inline thread_local dim3 threadIdx, blockIdx;
inline dim3 gridDim;

// The 32 lanes of the running warp are fibers on one thread: a shuffle stores
// the lane's value and yields; once every lane has yielded, each gets its
// partner's value and resumes.
struct Lane {
    ucontext_t ctx;
    float v, out;
    int o;
    bool done;
};
inline Lane g_lanes[32];
inline ucontext_t g_sched;
inline int g_cur = 0;
inline float __uint_as_float(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

namespace moe {
constexpr int kBlk = 32;
struct WsHeader {
    int status;
    unsigned done;
    int n_groups;
    unsigned bar, seq, pad0[3];
    unsigned long long wait_limit;
    int pad[54];
};
inline void record_error(int* status, int code) {
    std::atomic_ref<int> a(*status);
    int z = 0;
    a.compare_exchange_strong(z, code);
}
inline void pdl_wait() {}
inline void pdl_trigger() {}
inline uint4 ld16(const void* p) {
    if ((uintptr_t)p & 15u) { fprintf(stderr, "misaligned 16-byte load %p\n", p); std::abort(); }
    uint4 v; std::memcpy(&v, p, 16); return v;
}
inline uint4 ld_stream16(const void* p) { return ld16(p); }
inline uint4 ld_cg16(const void* p) { return ld16(p); }
inline float ld_cg_f32(const float* p) { return *p; }
inline int ld_cg_i32(const int* p) { return *p; }
inline float ldcg_f32(const float* p) { return *p; }
inline float ldcg_f32(const __nv_bfloat16* p) { return __uint_as_float((uint32_t)p->b << 16); }
inline float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
inline float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
inline float half2f(uint16_t h) {
    uint32_t s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    float v;
    if (e == 0) v = std::ldexp((float)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = std::ldexp((float)(m | 1024), (int)e - 25);
    return s ? -v : v;
}
template <typename T> inline float to_f32(T v);
template <> inline float to_f32<float>(float v) { return v; }
template <> inline float to_f32<__half>(__half v) { return half2f(v.b); }
inline float shfl_xor(float v, int o) {
    Lane& me = g_lanes[g_cur];
    me.v = v;
    me.o = o;
    swapcontext(&me.ctx, &g_sched);
    return g_lanes[g_cur].out;
}
inline float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += shfl_xor(v, o);
    return v;
}
inline float silu_mul(float g, float u) { return g / (1.0f + std::exp(-g)) * u; }

struct TopkParams {
    int T, E, k, norm_topk;
    const float* logits;
    const float* bias;
    int32_t* idx;
    float* w;
    float* probs;
};
inline cudaError_t launch_topk(const TopkParams&, cudaStream_t) { return cudaSuccess; }  // logits checked instead

template <typename P>
struct FiberJob {
    static inline void (*kern)(P);
    static inline const P* params;
    static void run() {
        kern(*params);
        g_lanes[g_cur].done = true;
    }
};

template <typename P>
cudaError_t launch(void (*kern)(P), dim3 grid, dim3 block, size_t, cudaStream_t, bool, P p) {
    gridDim = grid;
    const unsigned nw = block.x / 32;
    static std::vector<char> stacks(32 * 256 * 1024);
    FiberJob<P>::kern = kern;
    FiberJob<P>::params = &p;
    for (unsigned b = 0; b < grid.x; b++)
        for (unsigned w = 0; w < nw; w++) {
            for (int l = 0; l < 32; l++) {
                Lane& ln = g_lanes[l];
                ln.done = false;
                getcontext(&ln.ctx);
                ln.ctx.uc_stack.ss_sp = stacks.data() + (size_t)l * 256 * 1024;
                ln.ctx.uc_stack.ss_size = 256 * 1024;
                ln.ctx.uc_link = &g_sched;
                makecontext(&ln.ctx, (void (*)())FiberJob<P>::run, 0);
            }
            blockIdx = dim3(b);
            for (;;) {
                int ndone = 0;
                for (int l = 0; l < 32; l++) {
                    g_cur = l;
                    threadIdx = dim3(w * 32 + l);
                    if (!g_lanes[l].done) swapcontext(&g_sched, &g_lanes[l].ctx);
                    ndone += g_lanes[l].done;
                }
                if (ndone == 32) break;
                if (ndone != 0) { fprintf(stderr, "lanes diverged at a shuffle\n"); std::abort(); }
                for (int l = 0; l < 32; l++)
                    if (g_lanes[l].o != g_lanes[0].o) { fprintf(stderr, "lanes disagree on a shuffle\n"); std::abort(); }
                for (int l = 0; l < 32; l++) g_lanes[l].out = g_lanes[l ^ g_lanes[l].o].v;
            }
        }
    return cudaSuccess;
}

size_t shared_ws_bytes(int T, int F);
size_t preroute_ws_bytes(int T, int E, int H);
}  // namespace moe
