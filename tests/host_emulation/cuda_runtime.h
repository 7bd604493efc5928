// Test scaffolding: the CUDA runtime calls csrc/cache.cu makes, for compiling
// it as plain C++ on the CPU. Copies are immediate host copies and the stream
// and event calls do nothing, so the calls run in program order.
#pragma once
#include <cstddef>
#include <cstring>
typedef int cudaError_t;
constexpr int cudaSuccess = 0;
typedef void* cudaStream_t;
typedef void* cudaEvent_t;
enum cudaMemcpyKind { cudaMemcpyHostToDevice = 1, cudaMemcpyDeviceToHost = 2 };
inline int g_copies = 0;
inline cudaError_t cudaMemcpyAsync(void* d, const void* s, size_t n, cudaMemcpyKind, cudaStream_t) {
    std::memcpy(d, s, n);
    g_copies++;
    return cudaSuccess;
}
inline cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }
inline cudaError_t cudaStreamWaitEvent(cudaStream_t, cudaEvent_t, unsigned) { return cudaSuccess; }
inline cudaError_t cudaEventRecord(cudaEvent_t, cudaStream_t) { return cudaSuccess; }
