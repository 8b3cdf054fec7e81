// Host-side declarations shared by the C ABI (capi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace foak {

// Header at the start of a CE workspace.  `done` counts finished CTAs of the
// running call (the last one reduces the loss and sets it back to 0); `err`
// collects error bits of the running call (read and cleared by that last CTA).
struct CeWsHeader {
    unsigned int done;
    unsigned int err;
    unsigned int pad[62];
};
static_assert(sizeof(CeWsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kCeWsAlign = 256;

inline size_t ce_workspace_bytes(int64_t N) {
    const size_t rows = static_cast<size_t>(N < 0 ? 0 : N) * sizeof(float);
    return sizeof(CeWsHeader) + ((rows + kCeWsAlign - 1) / kCeWsAlign) * kCeWsAlign;
}

// Largest V the row kernel handles for an element size (2 or 4 bytes).
int64_t ce_rows_max_vocab(int elem_bytes);

// Forward (grad == false) or fused forward+backward in place (grad == true).
// row_loss must be non-null (caller buffer or the workspace's row area).
cudaError_t launch_ce_rows(bool grad, int elem_bytes, const void* x, void* dx, int64_t ld,
                           const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index, float g,
                           float denom, float* loss, float* lse, float* row_loss, int32_t* n_valid,
                           int32_t* err, CeWsHeader* ws, cudaStream_t stream);

cudaError_t launch_ce_backward(int elem_bytes, void* dx, const void* x, int64_t ld,
                               const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index,
                               const float* lse, const float* g_ptr, float denom, int32_t* err,
                               cudaStream_t stream);

// Streaming multiprocessor count of the current device (cached per device).
int device_sm_count();

}  // namespace foak
