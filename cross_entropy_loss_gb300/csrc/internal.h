// Host-side declarations shared by the C ABI (capi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace foak {

// Launch a kernel as a programmatic dependent of the work before it in the stream:
// it may be scheduled while the previous kernel finishes and must call
// griddep_wait() (common.cuh) before its first global-memory access.
template <typename... P, typename... A>
cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Header at the start of a CE workspace.  `done` counts finished CTAs of the
// running call (the last one reduces the loss and sets it back to 0); `err`
// collects error bits of the running call (read and cleared by that last CTA);
// `next` hands out the shared tail rows of the running call (reset to 0 by that
// last CTA too).
struct CeWsHeader {
    unsigned int done;
    unsigned int err;
    unsigned int next;
    unsigned int nvalid;  // label counts added by each CTA when they are counted on the way
    unsigned int nbad;
    unsigned int pad[59];
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
// row_loss must be non-null (caller buffer or the workspace's row area).  The
// denominator (when denom <= 0) and the error word's label check use
// count_labels[0, count_N) -- by default the rows' own labels; the chunked
// linear + CE passes the whole batch's labels so every chunk divides by the
// batch's n_valid.  The loss and n_valid outputs then describe this call's rows
// over that denominator.
cudaError_t launch_ce_rows(bool grad, int elem_bytes, const void* x, void* dx, int64_t ld,
                           const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index, float g,
                           float denom, float* loss, float* lse, float* row_loss, int32_t* n_valid,
                           int32_t* err, CeWsHeader* ws, cudaStream_t stream,
                           const int64_t* count_labels = nullptr, int64_t count_N = 0,
                           const int64_t* denom_dev = nullptr);

// Valid labels of labels[0, N) into *n_valid (int64, device) and, when err is
// given, FOAK_ERRBIT_LABEL_RANGE if some label is neither ignore_index nor in [0, V).
cudaError_t launch_count_valid(const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index, int64_t* n_valid,
                               int32_t* err, cudaStream_t stream);

// g = *g_ptr, or g_host when g_ptr is null; D = *denom_dev when given, else
// denom > 0 ? denom : the valid labels of labels[0, N).
cudaError_t launch_ce_backward(int elem_bytes, void* dx, const void* x, int64_t ld,
                               const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index,
                               const float* lse, const float* g_ptr, float denom, int32_t* err,
                               cudaStream_t stream, float g_host = 1.f, const int64_t* denom_dev = nullptr);

// Chunked linear + CE (linear_ce.cu): workspace bytes and the launch sequence.
size_t linear_ce_workspace_bytes(int64_t N, int64_t V, int64_t chunk);
// loss = (float64 sum of row_loss[0..N) in row order) / D, n_valid from labels, err
// = OR of the nerr words in chunk_err plus FOAK_ERRBIT_LABEL_RANGE for bad labels.
cudaError_t launch_rows_finalize(const float* row_loss, const int64_t* labels, int64_t N, int64_t V,
                                 int64_t ignore_index, float denom, const int32_t* chunk_err, int64_t nerr,
                                 float* loss, int32_t* n_valid, int32_t* err, cudaStream_t stream);
cudaError_t launch_linear_ce(const void* H, const void* W, const int64_t* labels, int64_t N, int64_t V, int64_t D,
                             int64_t ignore_index, int64_t chunk, float g, float denom, float* loss, void* dH,
                             float* dW, int32_t* n_valid, int32_t* err, void* workspace, cudaStream_t stream);

// Test hooks (capi.cu): the barrier-wait limit given to the row kernel, and a row
// whose slice the row kernel's producer skips (so a wait is sure to run out).
// RMSNorm (rmsnorm.cu): dgamma partials, up to 512 rows (CTAs or row groups) x D floats.
constexpr int kRmsGammaGroups = 128;
inline size_t rmsnorm_workspace_bytes(int64_t D) {
    return (static_cast<size_t>(512) * static_cast<size_t>(D) * 4 + 255) / 256 * 256;
}
cudaError_t launch_rmsnorm_fwd(int es, const void* X, int64_t ldx, const void* gamma, int64_t N, int64_t D,
                               float eps, void* Y, int64_t ldy, float* rstd, cudaStream_t s);
// dX (if N > 0) and, when dgamma is given, dgamma through `part` (rmsnorm_workspace_bytes(D)).
cudaError_t launch_rmsnorm_bwd(int es, const void* dY, int64_t lddy, const void* X, int64_t ldx, const void* gamma,
                               const float* rstd, int64_t N, int64_t D, void* dX, int64_t lddx, float* part,
                               float* dgamma, cudaStream_t s);

// RoPE (rope.cu): cos and sin planes of max_pos x d/2 floats, each 256-byte aligned.
size_t rope_cache_bytes(int64_t max_pos, int d);
cudaError_t launch_rope_cache(double base, int d, int64_t max_pos, void* cache, cudaStream_t s);
// X (H heads, token stride ldt) and, when X2 is non-null, X2 (H2 heads, ldt2) in one launch.
cudaError_t launch_rope_apply(int es, void* X, int64_t T, int H, int64_t ldt, void* X2, int H2, int64_t ldt2, int d,
                              const int64_t* positions, const void* cache, int64_t max_pos, bool inverse,
                              int32_t* err, cudaStream_t s);

uint64_t test_wait_limit_ns();
int64_t test_skip_load_row();
int32_t test_row_path();  // 0 automatic, 1 one pass (CTA / clusters), 2 two-pass streaming, 3 independent warps

// Streaming multiprocessor count of the current device (cached per device).
int device_sm_count();

}  // namespace foak
