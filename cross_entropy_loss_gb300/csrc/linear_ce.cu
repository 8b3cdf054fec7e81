// Chunked linear + cross-entropy: loss, dH and dW of CE(H W^T) without the full
// N x V logits -- the fused-linear / "chunked loss" form the FOAK pages name
// (LigerFusedLinearCrossEntropy, "Running Liger Kernel Benchmarks" on the
// fms-acceleration-foak 0.7.4 page; "add chunked loss" in the TODO of
// fms-acceleration PR #79).
//
// The batch's n_valid is counted once up front (unless the caller gives denom), so
// every chunk divides by the same D and the result does not depend on the chunk
// size.  Per chunk of rows [r0, r0 + C):
//   1. Z  = H_c W^T            tcgen05 GEMM, bf16 out (C x V scratch); its epilogue
//                              also reduces each row of each 128 x 256 output tile
//                              from the fp32 accumulator to (max, sum exp(z - max))
//                              and keeps the logit at the row's label
//   2. lse, row terms          one warp per row merges its tiles' pairs
//   3. dZ = (exp(Z - lse) - onehot) g / D   in place on Z, one streaming read and
//                              write per element (no row reduction)
//   4. dH_c = dZ W             tcgen05 GEMM, bf16 out into dH
//   5. dW (+)= dZ^T H          tcgen05 GEMM, fp32 out, once per group of
//                              kDeferChunks chunks (stored by the first group,
//                              added by TMA reduce for the others)
// and finally one CTA sums the per-row loss terms of all N rows (double-float, a
// fixed order) over the denominator.  The GEMMs run as grouped launches
// (launch_gemm_bf16_group): launch c holds step 1 of chunk c and step 4 of chunk
// c - 2 on one persistent grid, and its epilogue warps, idle until their first
// accumulator is ready, do step 3 of chunk c - 1 first (dH's 4 x 16 output units of
// 256 x 256 alone would leave 12 of the 76 SM pairs idle, and a separate dZ pass
// took 19 us per chunk).  Two groups' logits are resident.  Steps 1-2 are the GEMM-1
// epilogue statistics of the chunked loss; the softmax itself is rebuilt from Z and
// lse by step 3 rather than inside the producers of steps 4-5, whose operands would
// then each need an exponential at the tensor cores' rate.
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
    void* z;             // 2 kDeferChunks chunks x ldz bf16 (two dW groups)
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
    off += round256(static_cast<size_t>(std::min(2 * kDeferChunks * chunk, std::max<int64_t>(N, 1))) *
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
    // every error word starts at 0: the chunks' dZ passes and the GEMMs OR into theirs
    cudaError_t e = cudaMemsetAsync(ws.chunk_err, 0, static_cast<size_t>(nchunks + 1) * sizeof(int32_t), stream);
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
    auto rows_of = [&](int64_t c) { return static_cast<int>(std::min(chunk, N - c * chunk)); };
    // chunk c's logits live in slot c % (2 kDeferChunks): a dW group's chunks are adjacent
    auto z_of = [&](int64_t c) { return zbuf + (c % (2 * kDeferChunks)) * chunk * ldz; };
    auto z_desc = [&](int64_t c) {  // 1. Z = H_c W^T, with the epilogue statistics
        GemmDesc d = {};
        d.a = Hb + c * chunk * D;
        d.lda = D;
        d.b = W;
        d.ldb = D;
        d.M = rows_of(c);
        d.N = static_cast<int>(V);
        d.K = static_cast<int>(D);
        d.out = z_of(c);
        d.ldo = ldz;
        d.mode = kGemmOutBf16Stats;
        d.err = gemm_err;
        d.labels = labels + c * chunk;
        d.stats = ws.stats;
        d.stats_ld = tiles;
        d.zlab = ws.zlab;
        return d;
    };
    auto dh_desc = [&](int64_t c) {  // 4. dH_c = dZ_c W (W is [V][D]: MN-major as the [K][N] operand)
        GemmDesc d = {};
        d.a = z_of(c);
        d.lda = ldz;
        d.b = W;
        d.ldb = D;
        d.b_mn_major = true;
        d.M = rows_of(c);
        d.N = static_cast<int>(D);
        d.K = static_cast<int>(V);
        d.out = dHb + c * chunk * D;
        d.ldo = D;
        d.mode = kGemmOutBf16;
        d.err = gemm_err;
        return d;
    };
    auto dw_desc = [&](int64_t c_last) {  // 5. dW (+)= dZ_g^T H_g over the group ending at c_last
        const int64_t c0 = c_last - c_last % kDeferChunks;
        GemmDesc d = {};
        d.a = z_of(c0);  // dZ_g is [rows_g][V] = [K][M], H_g is [rows_g][D] = [K][N]
        d.lda = ldz;
        d.a_mn_major = true;
        d.b = Hb + c0 * chunk * D;
        d.ldb = D;
        d.b_mn_major = true;
        d.M = static_cast<int>(V);
        d.N = static_cast<int>(D);
        d.K = static_cast<int>(c_last * chunk + rows_of(c_last) - c0 * chunk);
        d.out = dW;
        d.ldo = D;
        d.mode = c0 == 0 ? kGemmOutF32 : kGemmOutF32Acc;
        d.err = gemm_err;
        return d;
    };
    auto side_of = [&](int64_t c) {  // 3. dZ_c = (softmax(Z_c) - onehot) * g / D in place
        GemmSideDz s = {};
        s.z = z_of(c);
        s.ldz = ldz;
        s.labels = labels + c * chunk;
        s.lse = ws.lse;
        s.rows = rows_of(c);
        s.V = static_cast<int>(V);
        s.ignore_index = ignore_index;
        s.g = g;
        s.denom = denom;
        s.denom_dev = denom_dev;
        s.err = ws.chunk_err + c;
        return s;
    };
    auto dz_alone = [&](int64_t c) {
        return launch_ce_backward(2, z_of(c), z_of(c), ldz, labels + c * chunk, rows_of(c), V, ignore_index, ws.lse,
                                  nullptr, denom, ws.chunk_err + c, stream, g, denom_dev);
    };
    // Launch c holds Z(c) and dH(c - 2), and its epilogue warps turn Z(c - 1) into dZ(c - 1)
    // before their first accumulator (they are idle then); the three touch three different
    // slots.  The lse of chunk c - 1 is in ws.lse from the kernel after launch c - 1.  A
    // group's dW, ready after the launch that finished its last dZ, rides in the next
    // launch (it reads its own half of the slots; Z(c) goes to the other half).
    int64_t dw_pending = -1;  // last chunk of a finished group whose dW is not launched yet
    for (int64_t c = 0; c < nchunks; ++c) {
        GemmDesc grp[3] = {z_desc(c), c >= 2 ? dh_desc(c - 2) : GemmDesc{}, GemmDesc{}};
        int np = c >= 2 ? 2 : 1;
        if (dw_pending >= 0) {
            grp[np++] = dw_desc(dw_pending);
            dw_pending = -1;
        }
        if (c >= 1) {
            const GemmSideDz side = side_of(c - 1);
            if (V % 8 == 0 && gemm_group_fits(grp, np)) {
                e = launch_gemm_bf16_group(grp, np, stream, &side);
            } else {  // single-CTA tiles or a ragged vocabulary: the dZ kernel by itself first
                e = dz_alone(c - 1);
                if (e == cudaSuccess) e = launch_gemm_bf16_group(grp, np, stream);
            }
        } else {
            e = launch_gemm_bf16_group(grp, np, stream);
        }
        if (e != cudaSuccess) return e;
        // 2. lse and row terms of chunk c's rows (into the batch's row_loss)
        const int rows = rows_of(c);
        e = launch_dependent(chunk_lse_kernel, dim3((rows + kMergeThreads / 32 - 1) / (kMergeThreads / 32)),
                             dim3(kMergeThreads), 0, stream, ws.stats, tiles, ws.zlab, labels + c * chunk, rows, V,
                             ignore_index, ws.lse, ws.row_loss + c * chunk);
        if (e != cudaSuccess) return e;
        // a group whose last dZ that launch wrote, unless it is the batch's last group:
        // its dW goes with the next launch, or by itself when there is none
        if (c >= 1 && (c - 1) % kDeferChunks == kDeferChunks - 1) {
            if (c + 1 < nchunks) {
                dw_pending = c - 1;
            } else {
                e = launch_gemm_bf16(dw_desc(c - 1), stream);
                if (e != cudaSuccess) return e;
            }
        }
    }
    if (nchunks > 0) {
        // the last chunk's dZ, then the last dH products and the last group's dW together
        const int64_t cl = nchunks - 1;
        e = dz_alone(cl);
        if (e != cudaSuccess) return e;
        GemmDesc fin[3];
        int nf = 0;
        if (cl >= 1) fin[nf++] = dh_desc(cl - 1);
        fin[nf++] = dh_desc(cl);
        fin[nf++] = dw_desc(cl);
        e = launch_gemm_bf16_group(fin, nf, stream);
        if (e != cudaSuccess) return e;
    }
    return launch_dependent(linear_ce_finalize, dim3(1), dim3(kFinThreads), 0, stream, ws.row_loss, labels, N, V,
                            ignore_index, denom, ws.chunk_err, nchunks + 1, loss, n_valid, err);
}

}  // namespace foak
