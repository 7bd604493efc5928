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
// wait limit), the E tagged logits and the k*F tagged activations.
constexpr int kNoAllocMaxE = 1024;
constexpr int kNoAllocMaxKF = 32768;
constexpr size_t kNoAllocHeader = 256;
constexpr size_t kNoAllocLogits = sizeof(uint64_t) * kNoAllocMaxE;
constexpr size_t kNoAllocH = sizeof(uint64_t) * kNoAllocMaxKF;
constexpr size_t kNoAllocBytes = kNoAllocHeader + kNoAllocLogits + kNoAllocH;  // 270,592 B
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
    if (router->E != E || router->D != D || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (D < kBlk || D % kBlk || F < kBlk || F % kBlk) return MOE_ERR_INVALID_ARG;
    if (E > kNoAllocMaxE || (long)k * F > kNoAllocMaxKF) return MOE_ERR_WORKSPACE;  // beyond the static scratch
    if (router->w_dtype != x_dtype || (x_dtype != MOE_F32 && x_dtype != MOE_BF16)) return MOE_ERR_UNSUPPORTED;
    if (experts->q != MOE_Q_INT8_SYM_B32 && experts->q != MOE_Q_INT4_SYM_B32) return MOE_ERR_UNSUPPORTED;
    if (experts->s_dtype != MOE_F32 && experts->s_dtype != MOE_F16) return MOE_ERR_UNSUPPORTED;
    const void* ptrs[8] = {router->W, x, experts->gate_q, experts->gate_s, experts->up_q,
                           experts->up_s, experts->down_q, experts->down_s};
    for (const void* p : ptrs)
        if (!al16(p)) return MOE_ERR_INVALID_ARG;
    if (!idx || !w || !al16(y) || (x_next && !al16(x_next))) return MOE_ERR_INVALID_ARG;
    if (router->bias && ((uintptr_t)router->bias & 3u)) return MOE_ERR_INVALID_ARG;

    const int qbits = experts->q == MOE_Q_INT8_SYM_B32 ? 8 : 4;
    FusedCommon fc = {};
    size_t smem = 0;
    int grid = 0;
    if (!fused_plan(E, D, F, k, qbits, experts->s_dtype == MOE_F16 ? 2 : 4, x_dtype == MOE_BF16 ? 2 : 4,
                    true, &fc, &smem, &grid))
        return MOE_ERR_UNSUPPORTED;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the scratch address below is the current device's: a stream of another
    // device would run the kernel against the wrong device's array
    if (s) {
        int cur = 0, sdev = 0;
        if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (sdev != cur) return MOE_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    // the status word must start at zero; the rest of the scratch is kept
    // consistent from one call to the next by the kernel itself (values are
    // tagged with the launch sequence number in the header)
    if (cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;

    unsigned char* base = static_cast<unsigned char*>(scratch);
    fc.nlayers = 1;
    fc.norm_topk = router->norm_topk ? 1 : 0;
    fc.hdr = reinterpret_cast<WsHeader*>(base);
    fc.logits = reinterpret_cast<uint64_t*>(base + kNoAllocHeader);
    fc.h = reinterpret_cast<uint64_t*>(base + kNoAllocHeader + kNoAllocLogits);
    fc.xex = nullptr;  // one layer: no layer output is exchanged
    FusedLayer ly = {};
    ly.W = router->W;
    ly.bias = router->bias;
    ly.x = x;
    ly.gate_q = experts->gate_q;
    ly.gate_s = experts->gate_s;
    ly.up_q = experts->up_q;
    ly.up_s = experts->up_s;
    ly.down_q = experts->down_q;
    ly.down_s = experts->down_s;
    ly.idx = idx;
    ly.w = w;
    ly.probs = probs;
    ly.y = y;
    ly.x_next = x_next;
    cudaError_t e = launch_fused(fc, &ly, qbits, experts->s_dtype == MOE_F16, x_dtype == MOE_BF16, grid, smem, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
