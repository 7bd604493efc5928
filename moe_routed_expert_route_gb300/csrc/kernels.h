// Kernel parameter blocks and launchers (internal to the library).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace moe {

// Launch with programmatic stream serialisation, so that a kernel may start its
// prologue while the previous kernel in the stream drains; every kernel calls
// griddepcontrol.wait before touching data the previous kernels produce.
template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    // static shared memory counts against the 48 KB default too: opt in early
    if (smem >= 16 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct RouterParams {
    int T, E, D, k, norm_topk;
    const void* W;          // [E][D] bf16 or fp32
    const float* bias;      // [E] or null
    const void* x;          // [T][D] bf16 or fp32
    float* logits;          // workspace [T][E]
    int32_t* idx;           // [T][k]
    float* w;               // [T][k]
    float* probs;           // [T][E] or null
    WsHeader* hdr;
    // fixed-point copy of x for the expert kernels (null: not produced)
    int8_t* xq_hi;
    uint8_t* xq_lo;
    float* xq_s;
    int qbits;
    // grouping of assignments by expert (null: not produced)
    int32_t* grp_expert;
    int32_t* grp_off;
    int32_t* assign;
};

struct ExpertParams {
    int T, E, D, F, k, qbits, s_f16;
    const void *gate_q, *gate_s, *up_q, *up_s, *down_q, *down_s;
    const int32_t* idx;     // [T][k]
    const float* w;         // [T][k]
    const void* x;          // [T][D] (residual source)
    int x_bf16;
    WsHeader* hdr;
    const int8_t* xq_hi;    // [T][D] fixed-point planes of x
    const uint8_t* xq_lo;
    const float* xq_s;      // [T][D/32]
    const int32_t* grp_expert;
    const int32_t* grp_off;
    const int32_t* assign;
    float* h;               // workspace [T*k][F]
    float* y;               // [T][D]
    void* x_next;           // [T][D] or null
    int max_groups;         // upper bound of distinct experts, sizes the grid
};

struct PrepParams {
    int T, E, D, k, qbits;
    const void* x;
    int x_bf16;
    const int32_t* idx;
    WsHeader* hdr;
    int8_t* xq_hi;
    uint8_t* xq_lo;
    float* xq_s;
    int32_t* grp_expert;
    int32_t* grp_off;
    int32_t* assign;
};

struct SubstituteParams {
    int T, E, k;
    const float* probs;
    const int32_t* idx_in;
    const float* w_in;
    const uint8_t* resident;
    float threshold;
    int32_t* idx_out;
    float* w_out;
    uint8_t* flag;
    float* mass;
};

// One layer of the persistent single-token layer kernel: its weights, its
// token and its outputs.
struct FusedLayer {
    const void* W;            // router [E][D], same dtype as x
    const float* bias;        // [E] or null
    const void* x;            // [D] input token
    const void *gate_q, *gate_s, *up_q, *up_s, *down_q, *down_s;
    const int32_t* idx_in;    // [k] routing when there is no router phase
    const float* w_in;
    const uint8_t* resident;  // [E] residency mask (substitution) or null
    int32_t* idx;             // [k] out: the router's top-k
    float* w;                 // [k] out: routing weights
    float* probs;             // [E] out or null
    int32_t* idx_used;        // [k] out or null: experts read after substitution
    uint8_t* sub_flag;        // [k] out or null
    float* sub_mass;          // [1] out or null
    float* y;                 // [D] out
    void* x_next;             // [D] out (x + y in x's dtype) or null
};

// Shape and workspace of a launch of the single-token layer kernel.
struct FusedCommon {
    int E, D, F, k, norm_topk, has_router, router_nseg, rows, nlayers, chain;
    float threshold;          // substitution threshold (with a residency mask)
    int pad;
    WsHeader* hdr;
    uint64_t* logits;         // workspace [E], tagged values
    uint64_t* h;              // workspace [k*F], tagged activations
    uint64_t* xex;            // workspace [D] (stacks only): a layer's x_next, tagged
};

constexpr int kFusedMaxGrid = 1024;  // CTAs of the layer kernel (<= SMs)
constexpr int kStackMax = 64;        // layers per launch of the layer kernel

template <int NL>
struct FusedArgs {
    FusedCommon c;
    FusedLayer L[NL];
};

// Router logits on the tensor cores: tile (mt, nt) = 128 token rows of x times
// 128 expert rows of Wr, both bf16 by TMA.
struct GemmParams {  // aligned like CUtensorMap
    CUtensorMap tmA;            // x [T][D] bf16, box {64, 128}, 128-byte swizzle
    CUtensorMap tmB0;           // Wr [E][D] bf16, box {64, 128}, 128-byte swizzle
    int K;                      // D
    int rows_per_ntile;         // 128
    int n_mtiles, m_total, n_ntiles;
    void* C;                    // fp32 logits [T][ldc]
    int ldc;
    WsHeader* hdr;
};

// Weight-stationary grouped expert projection (prefill): item i = (token tile
// i / nwb, weight block i % nwb); the A operand is a block of 128 dequantised
// weight rows, the B operand a tile of up to NT tokens' 16-bit rows.
struct EgParams {  // aligned like CUtensorMap
    CUtensorMap tmW0, tmW1;     // codes [rows][row bytes], box {64 or 32 bytes, 64 rows}, swizzled
                                // across the box's width (64 or 32 bytes)
    CUtensorMap tmX, tmXh;      // 16-bit B rows [positions][K], box {64, 128} / {64, 64}, 128-byte swizzle
    const void *S0, *S1;        // scales of W0 / W1 rows, [rows][K/32]
    int K;                      // reduction length
    int w_rows;                 // weight rows per expert in W0/W1
    int nwb;                    // weight blocks per expert
    const int32_t* tile_group;  // [tile] expert
    const int32_t* tile_m0;     // [tile] first position
    const int32_t* tile_n;      // [tile] positions in the tile
    const int* n_tiles_dev;     // number of tiles
    void* C;                    // fp16 H [pos][ldc] (SwiGLU) or fp32 Y [pos][ldc]
    int ldc;
    const int32_t* pexp;        // [pos] e: the B rows of position pos carry a factor 2^-e (SwiGLU:
                                // x rows; H is stored times 2^-2e) or 2^-2e (down: H rows)
    WsHeader* hdr;
};

// 2-D tensor map over a row-major matrix (dtype 0 = uint8, 1 = fp16, 2 = bf16),
// swizzle 0 (none) or 32, 64, 128 (bytes).
bool make_tmap_2d(CUtensorMap* m, int dtype, const void* base, unsigned long long inner, unsigned long long rows,
                  unsigned long long row_bytes, unsigned box_inner, unsigned box_rows, int swizzle);

struct TopkParams {
    int T, E, k, norm_topk;
    const float* logits;        // [T][E]
    const float* bias;          // [E] or null
    int32_t* idx;
    float* w;
    float* probs;               // [T][E] or null
};

constexpr int kPermChunk = 1024;  // assignments per histogram/placement CTA

struct PermParams {
    int n, k, E, nchunk;
    int tile_rows;              // positions per tile of the tile list
    const int32_t* idx;         // [n] expert of assignment i = t*k + r
    WsHeader* hdr;
    int32_t* chunk_cnt;         // [nchunk][E]
    int32_t* chunk_base;        // [nchunk][E]
    int32_t* cnt;               // [E]
    int32_t* off;               // [E+1]
    int32_t* group_end;         // [E]
    int32_t* counts_out;        // [E] or null
    int32_t* tile_group;        // [n/128 + E]
    int32_t* tile_m0;
    int32_t* tile_n;            // positions per tile (or null)
    int* n_mtiles;
    int32_t* perm_tok;          // [n] position -> token
    int32_t* perm_out;          // [n] position -> assignment id, or null
    int32_t* inv;               // [n] assignment -> position
};

struct CombineParams {
    int T, D, k;
    const int32_t* inv;
    const float* w;
    const float* Y;             // [n][D]
    float* y;                   // [T][D]
    const void* x;              // [T][D] residual source (x_next only)
    int x_bf16;
    void* x_next;               // [T][D] x + y in x's dtype, or null
};

cudaError_t launch_router_gemm(const GemmParams& p, cudaStream_t s);
cudaError_t launch_egemm(const EgParams& p, int qbits, bool s_f16, bool swiglu, int grid, cudaStream_t s);
constexpr int kEgTile = 128;  // token tile of the expert products
cudaError_t launch_topk(const TopkParams& p, cudaStream_t s);
cudaError_t launch_gather_f16(const void* x, bool x_bf16, const int32_t* perm_tok, int n, int D, void* Xp,
                              int32_t* pexp, cudaStream_t s);
cudaError_t launch_perm(const PermParams& p, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);

bool fused_plan(int E, int D, int F, int k, int qbits, int s_bytes, int x_bytes, bool has_router,
                FusedCommon* fc, size_t* smem, int* grid);
// nlayers = fc.nlayers entries of `layers` (<= kStackMax)
cudaError_t launch_fused(const FusedCommon& fc, const FusedLayer* layers, int qbits, bool s_f16, bool x_bf16,
                         int grid, size_t smem, cudaStream_t s);
int device_sm_count();
// workspace bytes of moe_shared_lora / moe_preroute (edge0.cu)
size_t shared_ws_bytes(int T, int F);
size_t preroute_ws_bytes(int T, int E, int H);
cudaError_t launch_router(const RouterParams& p, bool w_bf16, bool x_bf16, cudaStream_t s, bool pdl);
cudaError_t launch_prep(const PrepParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_experts(const ExpertParams& p, cudaStream_t s);
cudaError_t launch_substitute(const SubstituteParams& p, cudaStream_t s);
bool experts_supported(int T, int E, int D, int F, int k, int qbits);

}  // namespace moe
