// moe_layer_noalloc: the single-token layer without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run a
// layer: code that executes while a memory pool is frozen or being captured, a
// host runtime whose allocator is not reachable from the decode loop, or an
// embedding application that hands the library only its input and output
// buffers. For them this entry point keeps its scratch in a fixed, file-scope
// device array instead of a workspace. The array is part of the library's
// image: every GPU that loads the library holds it until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace moe {
namespace {

// Scratch of the layer kernel: header (status word, launch sequence number,
// completion counters), the E tagged logits and the k*F activations.
constexpr int kNoAllocMaxE = 1024;
constexpr int kNoAllocMaxKF = 32768;
constexpr size_t kNoAllocHeader = 256;
constexpr size_t kNoAllocLogits = sizeof(uint64_t) * kNoAllocMaxE;
constexpr size_t kNoAllocBytes = kNoAllocHeader + kNoAllocLogits + sizeof(float) * kNoAllocMaxKF;  // 139,520 B
static_assert(sizeof(WsHeader) == kNoAllocHeader, "header size");

// Zero-initialised at load time; shared by every call on the device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_dev_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once
// per device (host code only sees a host-side stand-in for the symbol).
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_dev_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_dev_ptr[dev] = p;
    }
    *out = g_dev_ptr[dev];
    return cudaSuccess;
}

bool al16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_layer_noalloc(const moe_router_t* router, const moe_experts_t* experts,
                                          const void* x, moe_dtype_t x_dtype, int32_t* idx, float* w,
                                          float* probs, float* y, void* x_next, void* stream) {
    if (!router || !experts) return MOE_ERR_INVALID_ARG;
    const int E = experts->E, D = experts->D, F = experts->F, k = router->k;
    if (router->E != E || router->D != D || k < 1 || k > E || k > 16) return MOE_ERR_INVALID_ARG;
    if (D < kBlk || D % kBlk || F < kBlk || F % kBlk) return MOE_ERR_INVALID_ARG;
    if (E > kNoAllocMaxE || (long)k * F > kNoAllocMaxKF) return MOE_ERR_WORKSPACE;  // beyond the static scratch
    if (router->w_dtype != x_dtype || (x_dtype != MOE_F32 && x_dtype != MOE_BF16)) return MOE_ERR_UNSUPPORTED;
    if (experts->q != MOE_Q_INT8_SYM_B32 && experts->q != MOE_Q_INT4_SYM_B32) return MOE_ERR_UNSUPPORTED;
    if (experts->s_dtype != MOE_F32 && experts->s_dtype != MOE_F16) return MOE_ERR_UNSUPPORTED;
    const void* ptrs[8] = {router->W, x, experts->gate_q, experts->gate_s, experts->up_q,
                           experts->up_s, experts->down_q, experts->down_s};
    for (const void* p : ptrs)
        if (!al16(p)) return MOE_ERR_INVALID_ARG;
    if (!idx || !w || !y || (x_next && !al16(x_next))) return MOE_ERR_INVALID_ARG;
    if (router->bias && ((uintptr_t)router->bias & 3u)) return MOE_ERR_INVALID_ARG;

    const int qbits = experts->q == MOE_Q_INT8_SYM_B32 ? 8 : 4;
    FusedParams fp = {};
    size_t smem = 0;
    int grid = 0;
    if (!fused_plan(E, D, F, k, qbits, experts->s_dtype == MOE_F16 ? 2 : 4, x_dtype == MOE_BF16 ? 2 : 4,
                    true, &fp, &smem, &grid))
        return MOE_ERR_UNSUPPORTED;

    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word must start at zero; the kernel's counters are kept
    // consistent from one call to the next by the kernel itself
    if (cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;

    unsigned char* base = static_cast<unsigned char*>(scratch);
    fp.E = E;
    fp.D = D;
    fp.F = F;
    fp.k = k;
    fp.has_router = 1;
    fp.norm_topk = router->norm_topk ? 1 : 0;
    fp.W = router->W;
    fp.bias = router->bias;
    fp.x = x;
    fp.gate_q = experts->gate_q;
    fp.gate_s = experts->gate_s;
    fp.up_q = experts->up_q;
    fp.up_s = experts->up_s;
    fp.down_q = experts->down_q;
    fp.down_s = experts->down_s;
    fp.idx = idx;
    fp.w = w;
    fp.probs = probs;
    fp.y = y;
    fp.x_next = x_next;
    fp.hdr = reinterpret_cast<WsHeader*>(base);
    fp.logits = reinterpret_cast<uint64_t*>(base + kNoAllocHeader);
    fp.h = reinterpret_cast<float*>(base + kNoAllocHeader + kNoAllocLogits);
    cudaError_t e = launch_fused(fp, qbits, experts->s_dtype == MOE_F16, x_dtype == MOE_BF16, grid, smem, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
