// Chunked linear + cross-entropy: loss, dH and dW of CE(H W^T) without the full
// N x V logits -- the fused-linear / "chunked loss" form the FOAK pages name
// (LigerFusedLinearCrossEntropy, "Running Liger Kernel Benchmarks" on the
// fms-acceleration-foak 0.7.4 page; "add chunked loss" in the TODO of
// fms-acceleration PR #79).
//
// The batch's n_valid is counted once up front (unless the caller gives denom), so
// every chunk divides by the same D and the result does not depend on the chunk
// size.  Then for each chunk of rows [r0, r0 + C):
//   1. Z  = H_c W^T            tcgen05 GEMM, bf16 out (C x V scratch); its epilogue
//                              also reduces each row of each 128 x 256 output tile
//                              from the fp32 accumulator to (max, sum exp(z - max))
//                              and keeps the logit at the row's label
//   2. lse, row terms          one warp per row merges its tiles' pairs
//   3. dZ = (exp(Z - lse) - onehot) g / D   the streaming backward kernel, in
//                              place on Z (one read, one write, no row reduction)
//   4. dH_c = dZ W             tcgen05 GEMM, bf16 out into dH
//   5. dW (+)= dZ^T H          tcgen05 GEMM, fp32 out, once per group of
//                              kDeferChunks chunks (stored by the first group,
//                              added by TMA reduce for the others)
// and finally one CTA sums the per-row loss terms of all N rows (double-float, a
// fixed order) over the denominator.  Step 4 of a chunk runs in one launch with step
// 1 of the next (two independent products on one persistent grid, see
// launch_gemm_bf16_group): dH's 4 x 16 output units of 256 x 256 would leave 12 of the
// 76 SM pairs idle for its whole run.  Only one group's Z lives at a time.  Steps 1-2
// are the GEMM-1 epilogue statistics of the chunked loss; the softmax itself is
// rebuilt from Z and lse by step 3 rather than inside the producers of steps 4-5,
// whose operands would then each need an exponential at the tensor cores' rate.
#include <algorithm>

#include "common.cuh"
#include "foak_ce.h"
#include "gemm_tc.h"
#include "internal.h"

namespace foak {

namespace {

constexpr int kFinThreads = 512;
// dW is updated once per group of this many chunks (one product with K = the
// group's rows): a quarter of the fp32 read-modify-write passes over dW and twice
// the k-blocks per output unit of two-chunk groups (chunked workload 4.27 -> 4.11 ms);
// only the group's logits are resident (4 x 65 MB at V = 32000, chunks of 1024).
constexpr int64_t kDeferChunks = 4;

inline size_t round256(size_t b) { return (b + 255) / 256 * 256; }

struct LinWs {
    int64_t* n_valid;    // the batch's valid labels (the denominator unless denom > 0)
    float* row_loss;     // N
    int32_t* chunk_err;  // one word per chunk's dZ pass, then one word for the GEMMs
    float2* stats;       // C x tiles per-tile (max, sum exp) of the chunk's rows
    float* zlab;         // C logits at the labels
    float* lse;          // C
    void* z;             // kDeferChunks chunks x ldz bf16
    size_t bytes;
};

int64_t lin_tiles(int64_t V) { return (V + kGemmTileN - 1) / kGemmTileN; }

LinWs lin_layout(void* base, int64_t N, int64_t V, int64_t chunk) {
    const int64_t nchunks = N > 0 ? (N + chunk - 1) / chunk : 0;
    const int64_t ldz = (V + 63) / 64 * 64;
    const size_t crows = static_cast<size_t>(std::min(chunk, std::max<int64_t>(N, 1)));
    LinWs w = {};
    size_t off = 0;
    char* b = static_cast<char*>(base);
    w.n_valid = reinterpret_cast<int64_t*>(b + off);
    off += 256;
    w.row_loss = reinterpret_cast<float*>(b + off);
    off += round256(static_cast<size_t>(N) * 4);
    w.chunk_err = reinterpret_cast<int32_t*>(b + off);
    off += round256(static_cast<size_t>(nchunks + 1) * 4);
    w.stats = reinterpret_cast<float2*>(b + off);
    off += round256(crows * static_cast<size_t>(lin_tiles(V)) * sizeof(float2));
    w.zlab = reinterpret_cast<float*>(b + off);
    off += round256(crows * 4);
    w.lse = reinterpret_cast<float*>(b + off);
    off += round256(crows * 4);
    w.z = b + off;
    off += round256(static_cast<size_t>(std::min(kDeferChunks * chunk, std::max<int64_t>(N, 1))) *
                    static_cast<size_t>(ldz) * 2);
    w.bytes = off;
    return w;
}

// loss = (double-float sum of the row terms, fixed order) / D; n_valid; error word.
__global__ void __launch_bounds__(kFinThreads) linear_ce_finalize(const float* __restrict__ row_loss,
                                                                  const int64_t* __restrict__ labels, int64_t N,
                                                                  int64_t V, int64_t ignore_index, float denom,
                                                                  const int32_t* chunk_err, int64_t nchunks,
                                                                  float* loss, int32_t* n_valid_out,
                                                                  int32_t* err_out) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    __shared__ int iscratch[2 * (kFinThreads / 32)];
    __shared__ DFloat dred[kFinThreads / 32];
    int n_valid = 0, n_bad = 0;
    count_labels(labels, N, V, ignore_index, iscratch, n_valid, n_bad);
    // the same 512-thread tree as the fused kernel's last CTA
    const DFloat tot = block_sum_terms<kFinThreads>(row_loss, N, dred);
    if (threadIdx.x == 0) {
        *loss = df_div(tot, denom > 0.f ? denom : static_cast<float>(n_valid));
        if (n_valid_out) *n_valid_out = n_valid;
        int32_t e = n_bad > 0 ? FOAK_ERRBIT_LABEL_RANGE : 0;
        for (int64_t c = 0; c < nchunks; ++c) e |= chunk_err[c];
        if (err_out) *err_out = e;
    }
}

constexpr int kMergeThreads = 256;  // one warp per row

// lse and the row term of each of a chunk's rows from its tiles' (max, sum exp) pairs.
__global__ void __launch_bounds__(kMergeThreads) chunk_lse_kernel(const float2* __restrict__ stats, int tiles,
                                                                  const float* __restrict__ zlab,
                                                                  const int64_t* __restrict__ labels, int rows,
                                                                  int64_t V, int64_t ignore_index,
                                                                  float* __restrict__ lse, float* __restrict__ row_loss) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    float m = kNegInf, s = 0.f;
    for (int t = lane; t < tiles; t += 32) {
        const float2 st = stats[static_cast<int64_t>(row) * tiles + t];
        ms_merge(m, s, st.x, st.y);
    }
    warp_ms_reduce(m, s);
    if (lane == 0) {
        const int64_t y = labels[row];
        const bool valid = y != ignore_index && y >= 0 && y < V;
        const float l = fmaf(lg2(s), kLn2, m);
        lse[row] = valid ? l : 0.f;
        row_loss[row] = valid ? l - zlab[row] : 0.f;
    }
}

}  // namespace

cudaError_t launch_rows_finalize(const float* row_loss, const int64_t* labels, int64_t N, int64_t V,
                                 int64_t ignore_index, float denom, const int32_t* chunk_err, int64_t nerr,
                                 float* loss, int32_t* n_valid, int32_t* err, cudaStream_t stream) {
    return launch_dependent(linear_ce_finalize, dim3(1), dim3(kFinThreads), 0, stream, row_loss, labels, N, V,
                            ignore_index, denom, chunk_err, nerr, loss, n_valid, err);
}

size_t linear_ce_workspace_bytes(int64_t N, int64_t V, int64_t chunk) {
    return lin_layout(nullptr, N, V, chunk).bytes;
}

cudaError_t launch_linear_ce(const void* H, const void* W, const int64_t* labels, int64_t N, int64_t V, int64_t D,
                             int64_t ignore_index, int64_t chunk, float g, float denom, float* loss, void* dH,
                             float* dW, int32_t* n_valid, int32_t* err, void* workspace, cudaStream_t stream) {
    const LinWs ws = lin_layout(workspace, N, V, chunk);
    const int64_t ldz = (V + 63) / 64 * 64;
    const int64_t nchunks = N > 0 ? (N + chunk - 1) / chunk : 0;
    int32_t* gemm_err = ws.chunk_err + nchunks;  // GEMM timeouts are OR-ed in here
    cudaError_t e = cudaMemsetAsync(gemm_err, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    if (nchunks == 0) {
        e = cudaMemsetAsync(dW, 0, static_cast<size_t>(V) * static_cast<size_t>(D) * 4, stream);
        if (e != cudaSuccess) return e;
    }
    // the batch's denominator, counted once for every chunk (unless the caller gives one)
    const int64_t* denom_dev = nullptr;
    if (!(denom > 0.f) && nchunks > 0) {
        e = launch_count_valid(labels, N, V, ignore_index, ws.n_valid, nullptr, stream);
        if (e != cudaSuccess) return e;
        denom_dev = ws.n_valid;
    }
    const int tiles = static_cast<int>(lin_tiles(V));
    const __nv_bfloat16* Hb = static_cast<const __nv_bfloat16*>(H);
    __nv_bfloat16* dHb = static_cast<__nv_bfloat16*>(dH);
    __nv_bfloat16* zbuf = static_cast<__nv_bfloat16*>(ws.z);
    // dH of a chunk goes out with the next chunk's Z in one launch (the 64 units of dH
    // alone leave 12 of the 76 SM pairs idle), and the last one with the last dW
    GemmDesc pend_dh = {};
    bool have_dh = false;
    for (int64_t c = 0; c < nchunks; ++c) {
        const int64_t r0 = c * chunk;
        const int rows = static_cast<int>(std::min(chunk, N - r0));
        const int64_t slot = c % kDeferChunks;  // this chunk's place in the group's Z buffer
        __nv_bfloat16* z = zbuf + slot * chunk * ldz;
        // 1. Z = H_c W^T
        GemmDesc g1 = {};
        g1.a = Hb + r0 * D;
        g1.lda = D;
        g1.a_mn_major = false;
        g1.b = W;
        g1.ldb = D;
        g1.b_mn_major = false;
        g1.M = rows;
        g1.N = static_cast<int>(V);
        g1.K = static_cast<int>(D);
        g1.out = z;
        g1.ldo = ldz;
        g1.mode = kGemmOutBf16Stats;
        g1.err = gemm_err;
        g1.labels = labels + r0;
        g1.stats = ws.stats;
        g1.stats_ld = tiles;
        g1.zlab = ws.zlab;
        {
            const GemmDesc grp[2] = {g1, pend_dh};  // Z(c) writes the other Z slot than dH(c-1) reads
            e = launch_gemm_bf16_group(grp, have_dh ? 2 : 1, stream);
            if (e != cudaSuccess) return e;
        }
        // 2. lse and row terms of the chunk's rows (into the batch's row_loss)
        e = launch_dependent(chunk_lse_kernel, dim3((rows + kMergeThreads / 32 - 1) / (kMergeThreads / 32)),
                             dim3(kMergeThreads), 0, stream, ws.stats, tiles, ws.zlab, labels + r0, rows, V,
                             ignore_index, ws.lse, ws.row_loss + r0);
        if (e != cudaSuccess) return e;
        // 3. dZ = (softmax(Z) - onehot) * g / D in place
        e = launch_ce_backward(2, z, z, ldz, labels + r0, rows, V, ignore_index, ws.lse, nullptr, denom,
                               ws.chunk_err + c, stream, g, denom_dev);
        if (e != cudaSuccess) return e;
        // 4. dH_c = dZ W     (W is [V][D]: MN-major as the [K][N] operand), launched later
        GemmDesc& g2 = pend_dh;
        g2 = GemmDesc{};
        g2.a = z;
        g2.lda = ldz;
        g2.a_mn_major = false;
        g2.b = W;
        g2.ldb = D;
        g2.b_mn_major = true;
        g2.M = rows;
        g2.N = static_cast<int>(D);
        g2.K = static_cast<int>(V);
        g2.out = dHb + r0 * D;
        g2.ldo = D;
        g2.mode = kGemmOutBf16;
        g2.err = gemm_err;
        have_dh = true;
        // 5. once the group is complete: dW (+)= dZ_g^T H_g over the group's rows
        //    (dZ_g is [rows_g][V] = [K][M], H_g is [rows_g][D] = [K][N])
        if (slot == kDeferChunks - 1 || c == nchunks - 1) {
            const int64_t g0 = (c - slot) * chunk;
            const int rows_g = static_cast<int>(r0 + rows - g0);
            GemmDesc g3 = {};
            g3.a = zbuf;
            g3.lda = ldz;
            g3.a_mn_major = true;
            g3.b = Hb + g0 * D;
            g3.ldb = D;
            g3.b_mn_major = true;
            g3.M = static_cast<int>(V);
            g3.N = static_cast<int>(D);
            g3.K = rows_g;
            g3.out = dW;
            g3.ldo = D;
            g3.mode = g0 == 0 ? kGemmOutF32 : kGemmOutF32Acc;
            g3.err = gemm_err;
            if (c == nchunks - 1) {
                const GemmDesc fin[2] = {pend_dh, g3};
                e = launch_gemm_bf16_group(fin, 2, stream);
                have_dh = false;
            } else {
                e = launch_gemm_bf16(g3, stream);
            }
            if (e != cudaSuccess) return e;
        }
    }
    return launch_dependent(linear_ce_finalize, dim3(1), dim3(kFinThreads), 0, stream, ws.row_loss, labels, N, V,
                            ignore_index, denom, ws.chunk_err, nchunks + 1, loss, n_valid, err);
}

}  // namespace foak
