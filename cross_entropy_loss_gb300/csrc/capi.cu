// C ABI of the library: argument checks, workspace layout, launches and the
// optional synchronous error check.  Declarations and their contracts are in
// include/foak_ce.h.
#include <algorithm>
#include <atomic>
#include <map>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "foak_ce.h"
#include "gemm_tc.h"
#include "internal.h"

namespace foak {

int device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

namespace {
std::atomic<uint64_t> g_wait_limit_ns{4000000000ull};
std::atomic<int64_t> g_skip_load_row{-1};
std::atomic<int32_t> g_row_path{0};
}  // namespace

uint64_t test_wait_limit_ns() { return g_wait_limit_ns.load(); }
int64_t test_skip_load_row() { return g_skip_load_row.load(); }
int32_t test_row_path() { return g_row_path.load(); }

namespace {

std::atomic<int> g_fail_launches{0};

bool take_injected_failure() {
    int n = g_fail_launches.load();
    while (n > 0) {
        if (g_fail_launches.compare_exchange_weak(n, n - 1)) return true;
    }
    return false;
}

bool sync_check_enabled() {
    const char* s = std::getenv("FOAK_SYNC_CHECK");
    return s && s[0] == '1';
}

int elem_bytes_of(int32_t dtype) {
    if (dtype == FOAK_BF16) return 2;
    if (dtype == FOAK_F32) return 4;
    return 0;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Vocabularies the chunked linear + CE calls take: 1024 columns of 256-column tiles
// (their logits slots, statistics and grouped unit lists are sized and tested up to it).
constexpr int64_t kLinearMaxVocab = 262144;

// Checks common to the row calls.
foak_status check_rows(const void* logits, int32_t dtype, int64_t ld, const int64_t* labels, int64_t N,
                       int64_t V, int* es) {
    *es = elem_bytes_of(dtype);
    if (*es == 0) return FOAK_ERR_UNSUPPORTED;
    if (N < 0 || V < 1 || ld < V) return FOAK_ERR_INVALID_ARG;
    if (N > 0x7fffffffLL) return FOAK_ERR_UNSUPPORTED;  // n_valid is int32
    if (V > ce_rows_max_vocab(*es)) return FOAK_ERR_UNSUPPORTED;
    if (N > 0 && (!logits || !labels)) return FOAK_ERR_INVALID_ARG;
    if (logits && !aligned(logits, static_cast<size_t>(*es))) return FOAK_ERR_INVALID_ARG;
    if (labels && !aligned(labels, 8)) return FOAK_ERR_INVALID_ARG;
    return FOAK_OK;
}

foak_status finish(cudaError_t e, int32_t* err, cudaStream_t stream) {
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return FOAK_ERR_CUDA;
    }
    if (!sync_check_enabled()) return FOAK_OK;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FOAK_ERR_CUDA;
    if (!err) return FOAK_OK;
    int32_t h = 0;
    if (cudaMemcpy(&h, err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FOAK_ERR_CUDA;
    if (h & FOAK_ERRBIT_TIMEOUT) return FOAK_ERR_TIMEOUT;
    if (h & FOAK_ERRBIT_LABEL_RANGE) return FOAK_ERR_LABEL_RANGE;
    return FOAK_OK;
}

foak_status rows_common(bool grad, const void* logits, int32_t dtype, int64_t ld, const int64_t* labels,
                        int64_t N, int64_t V, int64_t ignore_index, float g, float denom, float* loss,
                        float* lse, float* row_loss, int32_t* n_valid, int32_t* err, void* workspace,
                        size_t workspace_bytes, void* stream, const int64_t* denom_dev = nullptr) {
    int es = 0;
    foak_status st = check_rows(logits, dtype, ld, labels, N, V, &es);
    if (st != FOAK_OK) return st;
    if (!loss || !aligned(loss, 4)) return FOAK_ERR_INVALID_ARG;
    if ((lse && !aligned(lse, 4)) || (row_loss && !aligned(row_loss, 4)) || (n_valid && !aligned(n_valid, 4)) ||
        (err && !aligned(err, 4)))
        return FOAK_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, kCeWsAlign) || workspace_bytes < ce_workspace_bytes(N))
        return FOAK_ERR_WORKSPACE;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    CeWsHeader* ws = static_cast<CeWsHeader*>(workspace);
    float* rl = row_loss ? row_loss : reinterpret_cast<float*>(static_cast<char*>(workspace) + sizeof(CeWsHeader));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_ce_rows(grad, es, logits, grad ? const_cast<void*>(logits) : nullptr, ld, labels, N, V,
                                   ignore_index, g, denom, loss, lse, rl, n_valid, err, ws, s, nullptr, 0,
                                   denom_dev);
    if (e == cudaSuccess) e = cudaGetLastError();
    return finish(e, err, s);
}

// ---- host-buffer entry: layout, copy stream and events (one set per device)
constexpr int kHostMaxChunks = 32;
constexpr int64_t kHostChunkRows = 512;

struct HostWs {
    CeWsHeader* hdr;
    float* row_loss;     // N
    int32_t* chunk_err;  // kHostMaxChunks words, one per chunk launch
    float* chunk_loss;   // loss output of the chunk launches (unused)
    float* loss;
    int32_t* n_valid;
    int32_t* err;
};

size_t host_ws_bytes(int64_t N) {
    return sizeof(CeWsHeader) + (static_cast<size_t>(N) * 4 + 255) / 256 * 256 + 256;
}

HostWs host_layout(void* base, int64_t N) {
    char* b = static_cast<char*>(base);
    HostWs w;
    w.hdr = reinterpret_cast<CeWsHeader*>(b);
    w.row_loss = reinterpret_cast<float*>(b + sizeof(CeWsHeader));
    char* tail = b + sizeof(CeWsHeader) + (static_cast<size_t>(N) * 4 + 255) / 256 * 256;
    w.chunk_err = reinterpret_cast<int32_t*>(tail);
    w.chunk_loss = reinterpret_cast<float*>(tail + 4 * kHostMaxChunks);
    w.loss = w.chunk_loss + 1;
    w.n_valid = reinterpret_cast<int32_t*>(w.loss + 1);
    w.err = w.n_valid + 1;
    return w;
}

struct CopyLane {
    cudaStream_t cs = nullptr;
    cudaEvent_t ev[kHostMaxChunks + 1] = {};
};
std::mutex g_host_mu;  // serialises host-buffer calls: they share the lane of their device
std::map<int, CopyLane> g_lanes;

cudaError_t copy_lane(int dev, CopyLane** out) {
    CopyLane& l = g_lanes[dev];
    if (!l.cs) {
        cudaError_t e = cudaStreamCreateWithFlags(&l.cs, cudaStreamNonBlocking);
        if (e != cudaSuccess) return e;
        for (auto& ev : l.ev) {
            e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
    }
    *out = &l;
    return cudaSuccess;
}

// ---- RMSNorm entries
bool rows16(const void* p, int64_t ld, int es) { return aligned(p, 16) && (ld * es) % 16 == 0; }

inline size_t r256(size_t b) { return (b + 255) / 256 * 256; }

struct NormLinWs {
    void* lin;     // the chunked linear + CE workspace
    void* H;       // bf16 [N][D]: the normalised hidden states
    void* dH;      // bf16 [N][D]
    float* rstd;   // [N]
    float* part;   // dgamma partials
    size_t bytes;
};

NormLinWs norm_lin_layout(void* base, int64_t N, int64_t V, int64_t D, int64_t chunk) {
    char* b = static_cast<char*>(base);
    NormLinWs w;
    size_t off = 0;
    w.lin = b + off;
    off += r256(linear_ce_workspace_bytes(N, V, chunk));
    const size_t hd = r256(static_cast<size_t>(N) * static_cast<size_t>(D) * 2);
    w.H = b + off;
    off += hd;
    w.dH = b + off;
    off += hd;
    w.rstd = reinterpret_cast<float*>(b + off);
    off += r256(static_cast<size_t>(N) * 4);
    w.part = reinterpret_cast<float*>(b + off);
    off += rmsnorm_workspace_bytes(D);
    w.bytes = off;
    return w;
}

// Argument checks of one product (foak_gemm_bf16 / foak_gemm_bf16_group).
foak_status check_gemm(const foak_gemm_problem& q) {
    if (q.M < 0 || q.N < 0 || q.K < 0 || q.M > 0x7fffffffLL || q.N > 0x7fffffffLL || q.K > 0x7fffffffLL)
        return FOAK_ERR_INVALID_ARG;
    if (q.out_mode != FOAK_GEMM_BF16 && q.out_mode != FOAK_GEMM_F32 && q.out_mode != FOAK_GEMM_F32_ACC)
        return FOAK_ERR_INVALID_ARG;
    if (q.M == 0 || q.N == 0) return FOAK_OK;
    const int oes = q.out_mode == FOAK_GEMM_BF16 ? 2 : 4;
    if (!q.a || !q.b || !q.out || !aligned(q.a, 16) || !aligned(q.b, 16) || !aligned(q.out, 16))
        return FOAK_ERR_INVALID_ARG;
    if ((q.lda * 2) % 16 || (q.ldb * 2) % 16 || (q.ldo * oes) % 16 || q.ldo < q.N) return FOAK_ERR_INVALID_ARG;
    if (q.lda < (q.a_mn_major ? q.M : q.K) || q.ldb < (q.b_mn_major ? q.N : q.K)) return FOAK_ERR_INVALID_ARG;
    return FOAK_OK;
}

// An empty contraction: C = 0 (or unchanged when accumulating).
cudaError_t gemm_empty_k(const foak_gemm_problem& q, cudaStream_t s) {
    if (q.M == 0 || q.N == 0 || q.out_mode == FOAK_GEMM_F32_ACC) return cudaSuccess;
    const int oes = q.out_mode == FOAK_GEMM_BF16 ? 2 : 4;
    return cudaMemset2DAsync(q.out, static_cast<size_t>(q.ldo) * oes, 0, static_cast<size_t>(q.N) * oes,
                             static_cast<size_t>(q.M), s);
}

GemmDesc gemm_desc(const foak_gemm_problem& q, int32_t* err) {
    GemmDesc d = {};
    d.a = q.a;
    d.lda = q.lda;
    d.a_mn_major = q.a_mn_major != 0;
    d.b = q.b;
    d.ldb = q.ldb;
    d.b_mn_major = q.b_mn_major != 0;
    d.M = static_cast<int>(q.M);
    d.N = static_cast<int>(q.N);
    d.K = static_cast<int>(q.K);
    d.out = q.out;
    d.ldo = q.ldo;
    d.mode = static_cast<GemmOut>(q.out_mode);
    d.err = err;
    return d;
}

}  // namespace
}  // namespace foak

using namespace foak;

extern "C" {

const char* foak_status_string(int32_t status) {
    switch (status) {
        case FOAK_OK: return "FOAK_OK";
        case FOAK_ERR_INVALID_ARG: return "FOAK_ERR_INVALID_ARG: null, negative, misaligned or inconsistent argument";
        case FOAK_ERR_UNSUPPORTED: return "FOAK_ERR_UNSUPPORTED: dtype or size outside what the kernels handle";
        case FOAK_ERR_LABEL_RANGE: return "FOAK_ERR_LABEL_RANGE: a label was outside [0, V) and not ignore_index";
        case FOAK_ERR_WORKSPACE: return "FOAK_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case FOAK_ERR_CUDA: return "FOAK_ERR_CUDA: a CUDA call or kernel launch failed";
        case FOAK_ERR_TIMEOUT: return "FOAK_ERR_TIMEOUT: a device-side wait gave up";
        default: return "unknown foak_status";
    }
}

int32_t foak_abi_version(void) { return FOAK_CE_ABI_VERSION; }

int64_t foak_ce_max_vocab(int32_t dtype) {
    const int es = elem_bytes_of(dtype);
    return es ? ce_rows_max_vocab(es) : 0;
}

size_t foak_ce_workspace_size(int64_t N) { return ce_workspace_bytes(N); }

foak_status foak_ce_forward(const void* logits, int32_t dtype, int64_t ld, const int64_t* labels, int64_t N,
                            int64_t V, int64_t ignore_index, float denom, float* loss, float* lse,
                            float* row_loss, int32_t* n_valid, int32_t* err, void* workspace,
                            size_t workspace_bytes, void* stream) {
    return rows_common(false, logits, dtype, ld, labels, N, V, ignore_index, 1.0f, denom, loss, lse, row_loss,
                       n_valid, err, workspace, workspace_bytes, stream);
}

foak_status foak_ce_fwd_bwd(void* logits, int32_t dtype, int64_t ld, const int64_t* labels, int64_t N, int64_t V,
                            int64_t ignore_index, float g, float denom, float* loss, float* lse,
                            int32_t* n_valid, int32_t* err, void* workspace, size_t workspace_bytes,
                            void* stream) {
    return rows_common(true, logits, dtype, ld, labels, N, V, ignore_index, g, denom, loss, lse, nullptr,
                       n_valid, err, workspace, workspace_bytes, stream);
}

foak_status foak_ce_count_valid(const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index, int64_t* n_valid,
                                int32_t* err, void* stream) {
    if (N < 0 || V < 1 || !n_valid || !aligned(n_valid, 8)) return FOAK_ERR_INVALID_ARG;
    if (N > 0 && (!labels || !aligned(labels, 8))) return FOAK_ERR_INVALID_ARG;
    if (N > 0x7fffffffLL) return FOAK_ERR_UNSUPPORTED;
    if (err && !aligned(err, 4)) return FOAK_ERR_INVALID_ARG;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(launch_count_valid(labels, N, V, ignore_index, n_valid, err, s), err, s);
}

foak_status foak_ce_fwd_bwd_devdenom(void* logits, int32_t dtype, int64_t ld, const int64_t* labels, int64_t N,
                                     int64_t V, int64_t ignore_index, float g, const int64_t* denom_count,
                                     float* loss, float* lse, int32_t* n_valid, int32_t* err, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    if (!denom_count || !aligned(denom_count, 8)) return FOAK_ERR_INVALID_ARG;
    return rows_common(true, logits, dtype, ld, labels, N, V, ignore_index, g, 0.f, loss, lse, nullptr, n_valid, err,
                       workspace, workspace_bytes, stream, denom_count);
}

foak_status foak_ce_backward(void* dlogits, const void* logits, int32_t dtype, int64_t ld, const int64_t* labels,
                             int64_t N, int64_t V, int64_t ignore_index, const float* lse, const float* grad_out,
                             float denom, int32_t* err, void* stream) {
    int es = 0;
    foak_status st = check_rows(logits, dtype, ld, labels, N, V, &es);
    if (st != FOAK_OK) return st;
    if (N > 0 && (!dlogits || !lse)) return FOAK_ERR_INVALID_ARG;
    if (dlogits && !aligned(dlogits, static_cast<size_t>(es))) return FOAK_ERR_INVALID_ARG;
    // logits and dlogits share the row geometry: same offset modulo 16 bytes
    if (dlogits && logits &&
        (reinterpret_cast<uintptr_t>(dlogits) & 15u) != (reinterpret_cast<uintptr_t>(logits) & 15u))
        return FOAK_ERR_INVALID_ARG;
    if ((lse && !aligned(lse, 4)) || (grad_out && !aligned(grad_out, 4)) || (err && !aligned(err, 4)))
        return FOAK_ERR_INVALID_ARG;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        // nothing to compute; still report a clean error word
        cudaError_t e = err ? cudaMemsetAsync(err, 0, sizeof(int32_t), s) : cudaSuccess;
        return finish(e, err, s);
    }
    cudaError_t e = launch_ce_backward(es, dlogits, logits, ld, labels, N, V, ignore_index, lse, grad_out, denom,
                                       err, s);
    return finish(e, err, s);
}

size_t foak_linear_ce_workspace_size(int64_t N, int64_t V, int64_t D, int64_t chunk) {
    (void)D;
    if (N < 0 || V < 1 || chunk < 1) return 0;
    return linear_ce_workspace_bytes(N, V, chunk);
}

foak_status foak_linear_ce_chunked(const void* H, const void* W, const int64_t* labels, int64_t N, int64_t V,
                                   int64_t D, int64_t ignore_index, int64_t chunk, float g, float denom,
                                   float* loss, void* dH, float* dW, int32_t* n_valid, int32_t* err,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    if (N < 0 || V < 1 || D < 1 || chunk < 1) return FOAK_ERR_INVALID_ARG;
    if (N > 0x7fffffffLL || V > 0x7fffffffLL || D > 0x7fffffffLL) return FOAK_ERR_UNSUPPORTED;
    if (V > kLinearMaxVocab) return FOAK_ERR_UNSUPPORTED;
    if (D % 8) return FOAK_ERR_UNSUPPORTED;  // 16-byte rows for the tensor maps
    if (!W || !dW || !loss || !aligned(W, 16) || !aligned(dW, 16) || !aligned(loss, 4)) return FOAK_ERR_INVALID_ARG;
    if (N > 0 && (!H || !labels || !dH || !aligned(H, 16) || !aligned(dH, 16) || !aligned(labels, 8)))
        return FOAK_ERR_INVALID_ARG;
    if ((n_valid && !aligned(n_valid, 4)) || (err && !aligned(err, 4))) return FOAK_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, kCeWsAlign) || workspace_bytes < linear_ce_workspace_bytes(N, V, chunk))
        return FOAK_ERR_WORKSPACE;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(launch_linear_ce(H, W, labels, N, V, D, ignore_index, chunk, g, denom, loss, dH, dW, n_valid, err,
                                   workspace, s),
                  err, s);
}

size_t foak_rmsnorm_workspace_size(int64_t D) { return D < 1 ? 0 : rmsnorm_workspace_bytes(D); }

foak_status foak_rmsnorm_forward(const void* X, int32_t dtype, int64_t ldx, const void* gamma, int64_t N, int64_t D,
                                 float eps, void* Y, int64_t ldy, float* rstd, void* stream) {
    const int es = elem_bytes_of(dtype);
    if (!es) return FOAK_ERR_UNSUPPORTED;
    if (N < 0 || D < 8 || ldx < D || ldy < D || !(eps >= 0.f)) return FOAK_ERR_INVALID_ARG;
    if (D % 8) return FOAK_ERR_UNSUPPORTED;
    if (!gamma || !aligned(gamma, 16) || (rstd && !aligned(rstd, 4))) return FOAK_ERR_INVALID_ARG;
    if (N > 0 && (!X || !Y || !rows16(X, ldx, es) || !rows16(Y, ldy, es))) return FOAK_ERR_INVALID_ARG;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(launch_rmsnorm_fwd(es, X, ldx, gamma, N, D, eps, Y, ldy, rstd, s), nullptr, s);
}

foak_status foak_rmsnorm_backward(const void* dY, int64_t lddy, const void* X, int64_t ldx, const void* gamma,
                                  const float* rstd, int32_t dtype, int64_t N, int64_t D, void* dX, int64_t lddx,
                                  float* dgamma, void* workspace, size_t workspace_bytes, void* stream) {
    const int es = elem_bytes_of(dtype);
    if (!es) return FOAK_ERR_UNSUPPORTED;
    if (N < 0 || D < 8 || ldx < D || lddy < D || lddx < D) return FOAK_ERR_INVALID_ARG;
    if (D % 8) return FOAK_ERR_UNSUPPORTED;
    if (!gamma || !aligned(gamma, 16) || (dgamma && !aligned(dgamma, 4))) return FOAK_ERR_INVALID_ARG;
    if (N > 0 && (!dY || !X || !dX || !rstd || !rows16(dY, lddy, es) || !rows16(X, ldx, es) || !rows16(dX, lddx, es) ||
                  !aligned(rstd, 4)))
        return FOAK_ERR_INVALID_ARG;
    if (dgamma && (!workspace || !aligned(workspace, kCeWsAlign) || workspace_bytes < rmsnorm_workspace_bytes(D)))
        return FOAK_ERR_WORKSPACE;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(launch_rmsnorm_bwd(es, dY, lddy, X, ldx, gamma, rstd, N, D, dX, lddx, static_cast<float*>(workspace),
                                     dgamma, s),
                  nullptr, s);
}

size_t foak_rmsnorm_linear_ce_workspace_size(int64_t N, int64_t V, int64_t D, int64_t chunk) {
    if (N < 0 || V < 1 || D < 1 || chunk < 1) return 0;
    return norm_lin_layout(nullptr, N, V, D, chunk).bytes;
}

foak_status foak_rmsnorm_linear_ce_chunked(const void* X, const void* gamma, const void* W, const int64_t* labels,
                                           int64_t N, int64_t V, int64_t D, int64_t ignore_index, int64_t chunk,
                                           float eps, float g, float denom, float* loss, void* dX, float* dgamma,
                                           float* dW, int32_t* n_valid, int32_t* err, void* workspace,
                                           size_t workspace_bytes, void* stream) {
    if (N < 0 || V < 1 || D < 8 || chunk < 1 || !(eps >= 0.f)) return FOAK_ERR_INVALID_ARG;
    if (N > 0x7fffffffLL || V > 0x7fffffffLL || D > 0x7fffffffLL) return FOAK_ERR_UNSUPPORTED;
    if (V > kLinearMaxVocab || D % 8) return FOAK_ERR_UNSUPPORTED;
    if (!W || !dW || !loss || !gamma || !dgamma || !aligned(W, 16) || !aligned(dW, 16) || !aligned(loss, 4) ||
        !aligned(gamma, 16) || !aligned(dgamma, 4))
        return FOAK_ERR_INVALID_ARG;
    if (N > 0 && (!X || !labels || !dX || !aligned(X, 16) || !aligned(dX, 16) || !aligned(labels, 8)))
        return FOAK_ERR_INVALID_ARG;
    if ((n_valid && !aligned(n_valid, 4)) || (err && !aligned(err, 4))) return FOAK_ERR_INVALID_ARG;
    const NormLinWs w = norm_lin_layout(workspace, N, V, D, chunk);
    if (!workspace || !aligned(workspace, kCeWsAlign) || workspace_bytes < w.bytes) return FOAK_ERR_WORKSPACE;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // final norm (prologue) -> chunked LM head + CE -> norm backward (epilogue); H and dH stay on the device
    cudaError_t e = launch_rmsnorm_fwd(2, X, D, gamma, N, D, eps, w.H, D, w.rstd, s);
    if (e == cudaSuccess)
        e = launch_linear_ce(w.H, W, labels, N, V, D, ignore_index, chunk, g, denom, loss, w.dH, dW, n_valid, err,
                             w.lin, s);
    if (e == cudaSuccess) e = launch_rmsnorm_bwd(2, w.dH, D, X, D, gamma, w.rstd, N, D, dX, D, w.part, dgamma, s);
    return finish(e, err, s);
}

size_t foak_rope_cache_size(int64_t max_pos, int64_t d) {
    if (max_pos < 1 || d < 16 || d % 16 || d > (1 << 16)) return 0;
    return rope_cache_bytes(max_pos, static_cast<int>(d));
}

foak_status foak_rope_build_cache(double base, int64_t d, int64_t max_pos, void* cache, size_t cache_bytes,
                                  void* stream) {
    if (max_pos < 1 || !(base > 1.0)) return FOAK_ERR_INVALID_ARG;
    if (d < 16 || d % 16 || d > (1 << 16)) return FOAK_ERR_UNSUPPORTED;
    if (!cache || !aligned(cache, 256)) return FOAK_ERR_INVALID_ARG;
    if (cache_bytes < rope_cache_bytes(max_pos, static_cast<int>(d))) return FOAK_ERR_WORKSPACE;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(launch_rope_cache(base, static_cast<int>(d), max_pos, cache, s), nullptr, s);
}

foak_status foak_rope_apply(void* X, int32_t dtype, int64_t T, int64_t H, int64_t ldt, int64_t d,
                            const int64_t* positions, const void* cache, int64_t max_pos, int32_t inverse,
                            int32_t* err, void* stream) {
    const int es = elem_bytes_of(dtype);
    if (!es) return FOAK_ERR_UNSUPPORTED;
    if (d < 16 || d % 16 || d > (1 << 16)) return FOAK_ERR_UNSUPPORTED;
    if (T < 0 || H < 0 || H > 0x7fffffffLL || max_pos < 1 || ldt < H * d) return FOAK_ERR_INVALID_ARG;
    if (!cache || !aligned(cache, 256) || (err && !aligned(err, 4))) return FOAK_ERR_INVALID_ARG;
    if (T > 0 && H > 0 && (!X || !positions || !aligned(X, 16) || (ldt * es) % 16 || !aligned(positions, 8)))
        return FOAK_ERR_INVALID_ARG;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = err ? cudaMemsetAsync(err, 0, sizeof(int32_t), s) : cudaSuccess;
    if (e == cudaSuccess)
        e = launch_rope_apply(es, X, T, static_cast<int>(H), ldt, nullptr, 0, 0, static_cast<int>(d), positions, cache,
                              max_pos, inverse != 0, err, s);
    return finish(e, err, s);
}

foak_status foak_rope_apply_qk(void* Q, int64_t Hq, int64_t ldq, void* K, int64_t Hk, int64_t ldk, int32_t dtype,
                               int64_t T, int64_t d, const int64_t* positions, const void* cache, int64_t max_pos,
                               int32_t inverse, int32_t* err, void* stream) {
    const int es = elem_bytes_of(dtype);
    if (!es) return FOAK_ERR_UNSUPPORTED;
    if (d < 16 || d % 16 || d > (1 << 16)) return FOAK_ERR_UNSUPPORTED;
    if (T < 0 || Hq < 0 || Hk < 0 || Hq > 0x3fffffffLL || Hk > 0x3fffffffLL || max_pos < 1 || ldq < Hq * d ||
        ldk < Hk * d)
        return FOAK_ERR_INVALID_ARG;
    if (!cache || !aligned(cache, 256) || (err && !aligned(err, 4))) return FOAK_ERR_INVALID_ARG;
    if (T > 0 && (!positions || !aligned(positions, 8))) return FOAK_ERR_INVALID_ARG;
    if (T > 0 && Hq > 0 && (!Q || !aligned(Q, 16) || (ldq * es) % 16)) return FOAK_ERR_INVALID_ARG;
    if (T > 0 && Hk > 0 && (!K || !aligned(K, 16) || (ldk * es) % 16)) return FOAK_ERR_INVALID_ARG;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = err ? cudaMemsetAsync(err, 0, sizeof(int32_t), s) : cudaSuccess;
    if (e == cudaSuccess)
        e = launch_rope_apply(es, Hq > 0 ? Q : nullptr, T, static_cast<int>(Hq), ldq, Hk > 0 ? K : nullptr,
                              static_cast<int>(Hk), ldk, static_cast<int>(d), positions, cache, max_pos, inverse != 0,
                              err, s);
    return finish(e, err, s);
}

foak_status foak_gemm_bf16_group(const foak_gemm_problem* problems, int32_t n, int32_t* err, void* stream) {
    if (n < 0 || n > FOAK_GEMM_GROUP_MAX || (n > 0 && !problems)) return FOAK_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        const foak_status st = check_gemm(problems[i]);
        if (st != FOAK_OK) return st;
    }
    if (err && !aligned(err, 4)) return FOAK_ERR_INVALID_ARG;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmDesc d[FOAK_GEMM_GROUP_MAX];
    int nd = 0;
    cudaError_t e = cudaSuccess;
    for (int32_t i = 0; i < n && e == cudaSuccess; ++i) {
        const foak_gemm_problem& q = problems[i];
        if (q.M == 0 || q.N == 0) continue;
        if (q.K == 0) e = gemm_empty_k(q, s);
        else d[nd++] = gemm_desc(q, err);
    }
    if (e == cudaSuccess) e = launch_gemm_bf16_group(d, nd, s);
    return finish(e, err, s);
}

foak_status foak_gemm_bf16(const void* a, int64_t lda, int32_t a_mn_major, const void* b, int64_t ldb,
                           int32_t b_mn_major, int64_t M, int64_t N, int64_t K, void* out, int64_t ldo,
                           int32_t out_mode, int32_t* err, void* stream) {
    const foak_gemm_problem q = {a, lda, a_mn_major, b, ldb, b_mn_major, M, N, K, out, ldo, out_mode};
    const foak_status st = check_gemm(q);
    if (st != FOAK_OK || M == 0 || N == 0) return st;
    if (err && !aligned(err, 4)) return FOAK_ERR_INVALID_ARG;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return finish(gemm_empty_k(q, s), nullptr, s);
    return finish(launch_gemm_bf16(gemm_desc(q, err), s), err, s);
}

size_t foak_ce_host_workspace_size(int64_t N) { return N < 0 ? 0 : host_ws_bytes(N); }

foak_status foak_ce_fwd_bwd_host(const void* host_logits, int32_t dtype, int64_t ld, const int64_t* host_labels,
                                 int64_t N, int64_t V, int64_t ignore_index, float g, float denom,
                                 void* dev_logits, int64_t* dev_labels, float* host_loss, int32_t* host_n_valid,
                                 int32_t* host_err, void* workspace, size_t workspace_bytes, void* stream) {
    int es = 0;
    foak_status st = check_rows(dev_logits, dtype, ld, dev_labels, N, V, &es);
    if (st != FOAK_OK) return st;
    if (N > 0 && (!host_logits || !host_labels)) return FOAK_ERR_INVALID_ARG;
    if (!host_loss || (dev_logits && !aligned(dev_logits, 16))) return FOAK_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, kCeWsAlign) || workspace_bytes < host_ws_bytes(N)) return FOAK_ERR_WORKSPACE;
    if (take_injected_failure()) return FOAK_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return finish(e, nullptr, s);
    std::lock_guard<std::mutex> lock(g_host_mu);
    CopyLane* lane = nullptr;
    e = copy_lane(dev, &lane);
    if (e != cudaSuccess) return finish(e, nullptr, s);
    const HostWs w = host_layout(workspace, N);
    const int64_t nchunks =
        N == 0 ? 0 : std::min<int64_t>(kHostMaxChunks, std::max<int64_t>(1, (N + kHostChunkRows - 1) / kHostChunkRows));
    const int64_t per = nchunks ? (N + nchunks - 1) / nchunks : 0;
    const int64_t row_bytes = ld * es;
    // The copies start after the work already queued on `stream` (it may still use the device buffers).
    e = cudaEventRecord(lane->ev[0], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(lane->cs, lane->ev[0], 0);
    if (e == cudaSuccess && N > 0)
        e = cudaMemcpyAsync(dev_labels, host_labels, static_cast<size_t>(N) * 8, cudaMemcpyHostToDevice, lane->cs);
    for (int64_t c = 0; c < nchunks && e == cudaSuccess; ++c) {
        const int64_t r0 = c * per, r1 = std::min(N, r0 + per);
        if (r0 >= r1) break;
        const size_t bytes = static_cast<size_t>((r1 - r0 - 1) * ld + V) * es;  // up to the last row's V-th element
        e = cudaMemcpyAsync(static_cast<char*>(dev_logits) + r0 * row_bytes,
                            static_cast<const char*>(host_logits) + r0 * row_bytes, bytes, cudaMemcpyHostToDevice,
                            lane->cs);
        if (e == cudaSuccess) e = cudaEventRecord(lane->ev[1 + c], lane->cs);
    }
    // Each chunk is swept as soon as it has landed; every chunk divides by the n_valid of all N labels.
    int64_t launched = 0;
    for (int64_t c = 0; c < nchunks && e == cudaSuccess; ++c) {
        const int64_t r0 = c * per, r1 = std::min(N, r0 + per);
        if (r0 >= r1) break;
        e = cudaStreamWaitEvent(s, lane->ev[1 + c], 0);
        char* x = static_cast<char*>(dev_logits) + r0 * row_bytes;
        if (e == cudaSuccess)
            e = launch_ce_rows(true, es, x, x, ld, dev_labels + r0, r1 - r0, V, ignore_index, g, denom, w.chunk_loss,
                               nullptr, w.row_loss + r0, nullptr, w.chunk_err + c, w.hdr, s, dev_labels, N);
        ++launched;
    }
    if (e == cudaSuccess)
        e = launch_rows_finalize(w.row_loss, dev_labels, N, V, ignore_index, denom, w.chunk_err, launched, w.loss,
                                 w.n_valid, w.err, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(host_loss, w.loss, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && host_n_valid) e = cudaMemcpyAsync(host_n_valid, w.n_valid, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && host_err) e = cudaMemcpyAsync(host_err, w.err, 4, cudaMemcpyDeviceToHost, s);
    return finish(e, w.err, s);
}

void foak_test_fail_next_launches(int32_t count) { g_fail_launches.store(count < 0 ? 0 : count); }

void foak_test_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns == 0 ? 4000000000ull : ns); }

void foak_test_skip_row_load(int64_t row) { g_skip_load_row.store(row < 0 ? -1 : row); }

int32_t foak_test_gemm_group_schedule(const int64_t* mnk, int32_t n, int32_t pairs, int32_t* start, int32_t* ent,
                                      int32_t ent_cap) {
    return gemm_group_schedule(mnk, n, pairs, start, ent, ent_cap);
}

void foak_test_set_row_path(int32_t path) { g_row_path.store(path >= 1 && path <= 3 ? path : 0); }

}  // extern "C"
