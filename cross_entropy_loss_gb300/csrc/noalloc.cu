// Fused forward+backward for callers that may not allocate device memory.
//
// Some callers cannot hand this library a workspace: code on a latency-critical
// path where cudaMalloc/cudaFree would synchronise the whole device, or a plugin
// inside a runtime that owns every byte of device memory and forbids allocations
// while it executes.  foak_ce_fwd_bwd_noalloc serves them: it runs the same fused
// row kernel as foak_ce_fwd_bwd, but its scratch (the call's 256-byte header and
// one float per row for the loss terms) lives in the file-scope array below,
// which the CUDA runtime places in device memory when the library's module is
// loaded on a device and keeps there until the process exits.  Nothing is
// allocated or freed per call.
#include <mutex>

#include "foak_ce.h"
#include "internal.h"

namespace foak {
namespace {

constexpr size_t kNoallocBytes = sizeof(CeWsHeader) + static_cast<size_t>(FOAK_CE_NOALLOC_MAX_ROWS) * sizeof(float);

// Shared by every call on a device; holds whatever the last call left in it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  The host-side
// symbol is only a stand-in, so the address is looked up once per device (the
// first call on that device does it) and cached.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace foak

using namespace foak;

extern "C" foak_status foak_ce_fwd_bwd_noalloc(void* logits, int32_t dtype, int64_t ld, const int64_t* labels,
                                               int64_t N, int64_t V, int64_t ignore_index, float g, float denom,
                                               float* loss, float* lse, int32_t* n_valid, int32_t* err,
                                               void* stream) {
    if (N > FOAK_CE_NOALLOC_MAX_ROWS) return FOAK_ERR_WORKSPACE;  // larger batches need foak_ce_fwd_bwd
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) {
        (void)cudaGetLastError();
        return FOAK_ERR_CUDA;
    }
    // The kernel's completion counter and error word must start at zero; the row
    // area is fully rewritten by every call.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, sizeof(CeWsHeader), s) != cudaSuccess) {
        (void)cudaGetLastError();
        return FOAK_ERR_CUDA;
    }
    return foak_ce_fwd_bwd(logits, dtype, ld, labels, N, V, ignore_index, g, denom, loss, lse, n_valid, err,
                           scratch, kNoallocBytes, stream);
}
