// Host interface of the tcgen05 GEMM used by the chunked linear + cross-entropy.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace foak {

enum GemmOut : int {
    kGemmOutBf16 = 0,    // C = A * B^T, stored as bf16
    kGemmOutF32 = 1,     // C = A * B^T, stored as fp32
    kGemmOutF32Acc = 2,  // C += A * B^T in fp32 (read-modify-write)
    kGemmOutBf16Stats = 3,  // as kGemmOutBf16, plus per-(row, 256-column tile) softmax statistics of
                            // the fp32 accumulator: stats[row * stats_ld + tile] = (max, sum exp(c - max))
                            // over the tile's columns, and zlab[row] = C[row][labels[row]] when the
                            // label is a column of the product (rows of C are the labels' rows)
};

// C[M x N] (+)= A[M x K] * B[N x K]^T, bf16 operands, fp32 accumulation.
// An operand is K-major when stored row-major as [rows][K] (row stride ld) and
// MN-major when stored row-major as [K][rows] (row stride ld).  Pointers and row
// strides must be 16-byte aligned; C is row-major with row stride ldo.
struct GemmDesc {
    const void* a;
    int64_t lda;
    bool a_mn_major;
    const void* b;
    int64_t ldb;
    bool b_mn_major;
    int M, N, K;
    void* out;
    int64_t ldo;
    GemmOut mode;
    int32_t* err;  // device error word for wait timeouts (may be null)
    // kGemmOutBf16Stats only
    const int64_t* labels;
    float2* stats;
    int stats_ld;
    float* zlab;
};

// Output tiles of the GEMM are kGemmTileN columns wide (the statistics' tile width).
constexpr int kGemmTileN = 256;

cudaError_t launch_gemm_bf16(const GemmDesc& d, cudaStream_t stream);

// Streaming work the epilogue warps of a grouped launch do before their first
// accumulator is ready (they are idle then): the cross-entropy gradient of a chunk's
// bf16 logits in place, z <- (exp(z - lse_row) - [col == label_row]) * g / D, rows of
// ignored labels (or labels outside [0, V), which set FOAK_ERRBIT_LABEL_RANGE in err)
// zero-filled.  V % 8 == 0 and 16-byte aligned rows (gemm_side_fits).  The same
// arithmetic, element for element, as the separate backward kernel.
struct GemmSideDz {
    void* z;                   // bf16 [rows][ldz]
    int64_t ldz;
    const int64_t* labels;     // [rows]
    const float* lse;          // [rows], natural log
    int rows;
    int V;
    int64_t ignore_index;
    float g;
    float denom;               // used when denom_dev is null
    const int64_t* denom_dev;  // the denominator as an int64 in device memory, or null
    int32_t* err;              // OR-ed with FOAK_ERRBIT_LABEL_RANGE; may be null
};

// Up to three independent products in one persistent launch of the CTA-pair kernel
// (every product with M > 128): the clusters take a list of (product, output unit)
// entries balanced by estimated cost, longest first.  No product may write what another
// reads.  Other cases are launched one product after another, in order.  The error word
// of the first product receives every timeout.
cudaError_t launch_gemm_bf16_group(const GemmDesc* d, int n, cudaStream_t stream, const GemmSideDz* side = nullptr);

// Whether launch_gemm_bf16_group runs these products as one grouped launch (and so can
// take a side job): every product on CTA pairs (M > 128), at most 8192 units.
bool gemm_group_fits(const GemmDesc* d, int n);

// The grouped launch's unit list for products of shapes mnk[3 q ..] on `pairs` SM
// pairs (host only); returns the clusters used or -1.
int gemm_group_schedule(const int64_t* mnk, int n, int pairs, int32_t* start, int32_t* ent, int ent_cap);

}  // namespace foak
