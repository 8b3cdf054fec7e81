// Pieces shared by the row-wise cross-entropy kernels (one CTA or one cluster
// per row, and one CTA streaming a long row in two passes): launch parameters,
// row geometry for rows that do not start on a 16-byte boundary, the packed
// per-thread arithmetic, and the last-CTA loss reduction.
#pragma once

#include "common.cuh"
#include "foak_ce.h"
#include "internal.h"

namespace foak {
// A CTA's slice of a row is at most 4096 16-byte vectors (64 KB), held in
// registers as 8 vectors per thread (512 threads) or 4 (1024 threads).
constexpr int kRowSliceVecMax = 4096;
constexpr int kRowMaxStages = 4;
constexpr int kRowMaxCluster = 8;
constexpr int kMaxScalars = 7;                        // head or tail: < 16 bytes of bf16
constexpr uint32_t kBulkChunk = 32768;
constexpr int kLabCache = 1024;                       // labels of a CTA's first rows kept in smem
constexpr int kTailMax = 2048;                        // shared tail rows handed out at run time
constexpr int kTailIgnoredDiv = 16;                   // ... when at least N / 16 rows are ignored
constexpr size_t kSmemBudget = 227 * 1024 - 28 * 1024; // dynamic smem left after static use

// Launch attribute: the kernel may start while the previous kernel of its stream is
// still running (it touches only shared memory until griddep_wait()).
inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

struct CeRowParams {
    const char* x;
    char* dx;
    int64_t ld;
    const int64_t* labels;
    int64_t N, V, ignore_index;
    float g, denom;
    const int64_t* denom_dev;  // if set: the denominator, read from device memory (overrides denom)
    float* loss;
    float* lse;
    float* row_loss;
    int32_t* n_valid;
    int32_t* err;
    CeWsHeader* ws;
    const int64_t* count_labels;  // labels whose valid count is the denominator (the batch's)
    int64_t count_N;
    uint64_t wait_ns;        // limit of every shared-memory barrier wait
    int64_t skip_load_row;   // test hook: this row's slice is never loaded (-1: none)
    int l2_hint;             // two-pass kernel: 0 none, 1 pass 1 evict_last + pass 2 evict_first, 2 pass 2 evict_first
    int tail_rounds;     // single-CTA rows: rows below tail_rounds * gridDim.x go round-robin, the
                         // valid rows from there on are handed out one at a time; -1: all round-robin
    int k;               // CTAs per row (cluster size)
    int per;             // vectors per CTA slice
    int stages;          // rows in flight per CTA
    uint32_t stage_bytes;
};

struct RowGeom {
    int h;       // scalar head elements before the first 16-byte boundary
    int64_t nb;  // 16-byte vectors
    int t;       // scalar tail elements
};

template <int ES>
__device__ __forceinline__ RowGeom row_geom(const char* rowp, int64_t V) {
    constexpr int EPV = 16 / ES;
    RowGeom g;
    int h = static_cast<int>(((16u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(rowp)) & 15u)) & 15u) / ES);
    if (h > V) h = static_cast<int>(V);
    g.h = h;
    g.nb = (V - h) / EPV;
    g.t = static_cast<int>(V - h - g.nb * EPV);
    return g;
}

template <int ES>
__device__ __forceinline__ float load_scalar(const char* p) {
    if constexpr (ES == 2) return bf16_lo(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)));
    else return *reinterpret_cast<const float*>(p);
}

template <int ES>
__device__ __forceinline__ void store_scalar(char* p, float v) {
    if constexpr (ES == 2) *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
    else *reinterpret_cast<float*>(p) = v;
}

// Per-thread arithmetic on the thread's slice (VPT 16-byte vectors).  Vectors
// beyond the slice hold -inf, which no max picks and whose exp is 0, so the
// loops run without predicates.
template <int ES>
struct RowMath;

template <>
struct RowMath<2> {  // bf16: 8 elements per vector, handled as 4 packed pairs
    static __device__ __forceinline__ uint4 pad() { return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u); }
    template <int VPT>
    static __device__ __forceinline__ float vmax(const uint4 (&v)[VPT]) {
        uint32_t a = v[0].x, b = v[0].y, c = v[0].z, d = v[0].w;
#pragma unroll
        for (int i = 1; i < VPT; ++i) {
            a = bf16x2_max(a, v[i].x);
            b = bf16x2_max(b, v[i].y);
            c = bf16x2_max(c, v[i].z);
            d = bf16x2_max(d, v[i].w);
        }
        const uint32_t m = bf16x2_max(bf16x2_max(a, b), bf16x2_max(c, d));
        return fmaxf(bf16_lo(m), bf16_hi(m));
    }
    // sum over the slice of 2^(x*log2e - mb)
    template <int VPT>
    static __device__ __forceinline__ float vsum(const uint4 (&v)[VPT], float mb) {
        const f32x2_t L = f2_pack(kLog2e, kLog2e), C = f2_pack(-mb, -mb);
        f32x2_t a = 0, b = 0, c = 0, d = 0;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            a = f2_add(a, f2_ex2(f2_fma(bf16x2_to_f2(v[i].x), L, C)));
            b = f2_add(b, f2_ex2(f2_fma(bf16x2_to_f2(v[i].y), L, C)));
            c = f2_add(c, f2_ex2(f2_fma(bf16x2_to_f2(v[i].z), L, C)));
            d = f2_add(d, f2_ex2(f2_fma(bf16x2_to_f2(v[i].w), L, C)));
        }
        float lo, hi;
        f2_unpack(f2_add(f2_add(a, b), f2_add(c, d)), lo, hi);
        return lo + hi;
    }
    // 2^(x*log2e - c) for every element, optionally times S
    template <bool MUL>
    static __device__ __forceinline__ uint4 vexp(const uint4& v, f32x2_t L, f32x2_t C, f32x2_t S) {
        uint4 o;
        f32x2_t t0 = f2_ex2(f2_fma(bf16x2_to_f2(v.x), L, C));
        f32x2_t t1 = f2_ex2(f2_fma(bf16x2_to_f2(v.y), L, C));
        f32x2_t t2 = f2_ex2(f2_fma(bf16x2_to_f2(v.z), L, C));
        f32x2_t t3 = f2_ex2(f2_fma(bf16x2_to_f2(v.w), L, C));
        if (MUL) {
            t0 = f2_mul(t0, S);
            t1 = f2_mul(t1, S);
            t2 = f2_mul(t2, S);
            t3 = f2_mul(t3, S);
        }
        o.x = f2_to_bf16x2(t0);
        o.y = f2_to_bf16x2(t1);
        o.z = f2_to_bf16x2(t2);
        o.w = f2_to_bf16x2(t3);
        return o;
    }
};

template <>
struct RowMath<4> {  // fp32: 4 elements per vector, 2 packed pairs
    static __device__ __forceinline__ uint4 pad() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
    template <int VPT>
    static __device__ __forceinline__ float vmax(const uint4 (&v)[VPT]) {
        float a = __uint_as_float(v[0].x), b = __uint_as_float(v[0].y);
        float c = __uint_as_float(v[0].z), d = __uint_as_float(v[0].w);
#pragma unroll
        for (int i = 1; i < VPT; ++i) {
            a = fmaxf(a, __uint_as_float(v[i].x));
            b = fmaxf(b, __uint_as_float(v[i].y));
            c = fmaxf(c, __uint_as_float(v[i].z));
            d = fmaxf(d, __uint_as_float(v[i].w));
        }
        return fmaxf(fmaxf(a, b), fmaxf(c, d));
    }
    template <int VPT>
    static __device__ __forceinline__ float vsum(const uint4 (&v)[VPT], float mb) {
        const f32x2_t L = f2_pack(kLog2e, kLog2e), C = f2_pack(-mb, -mb);
        f32x2_t a = 0, b = 0, c = 0, d = 0;
#pragma unroll
        for (int i = 0; i < VPT; i += 2) {
            a = f2_add(a, f2_ex2(f2_fma(f2_pack(__uint_as_float(v[i].x), __uint_as_float(v[i].y)), L, C)));
            b = f2_add(b, f2_ex2(f2_fma(f2_pack(__uint_as_float(v[i].z), __uint_as_float(v[i].w)), L, C)));
            c = f2_add(c, f2_ex2(f2_fma(f2_pack(__uint_as_float(v[i + 1].x), __uint_as_float(v[i + 1].y)), L, C)));
            d = f2_add(d, f2_ex2(f2_fma(f2_pack(__uint_as_float(v[i + 1].z), __uint_as_float(v[i + 1].w)), L, C)));
        }
        float lo, hi;
        f2_unpack(f2_add(f2_add(a, b), f2_add(c, d)), lo, hi);
        return lo + hi;
    }
    template <bool MUL>
    static __device__ __forceinline__ uint4 vexp(const uint4& v, f32x2_t L, f32x2_t C, f32x2_t S) {
        f32x2_t t0 = f2_ex2(f2_fma(f2_pack(__uint_as_float(v.x), __uint_as_float(v.y)), L, C));
        f32x2_t t1 = f2_ex2(f2_fma(f2_pack(__uint_as_float(v.z), __uint_as_float(v.w)), L, C));
        if (MUL) {
            t0 = f2_mul(t0, S);
            t1 = f2_mul(t1, S);
        }
        uint4 o;
        float a, b;
        f2_unpack(t0, a, b);
        o.x = __float_as_uint(a);
        o.y = __float_as_uint(b);
        f2_unpack(t1, a, b);
        o.z = __float_as_uint(a);
        o.w = __float_as_uint(b);
        return o;
    }
};

// The mean's denominator D: a count in device memory (the data-parallel total of
// valid tokens, all-reduced by the caller), else the caller's denom, else this
// call's own count of valid labels.
__device__ __forceinline__ float row_denominator(const CeRowParams& p, int n_valid) {
    if (p.denom_dev) return static_cast<float>(__ldg(p.denom_dev));
    return p.denom > 0.f ? p.denom : static_cast<float>(n_valid);
}

// One CTA per row, the row streamed through shared memory in 64 KB chunks
// twice (log-sum-exp, then gradient): for rows longer than one CTA's slice.
cudaError_t launch_ce_rows_long(bool grad, int elem_bytes, const CeRowParams& base, cudaStream_t stream);

// Aligned rows of at most one 64 KB slice (V * elem_bytes a multiple of 16, every
// row on a 16-byte boundary, dlogits in place): one CTA per SM, its 16 warps each
// moving a 4 KB region of every row on their own.
bool ce_rows_warp_fits(int elem_bytes, int64_t V);
cudaError_t launch_ce_rows_warp(bool grad, int elem_bytes, const CeRowParams& base, cudaStream_t stream);

// End of a row kernel: every CTA counts itself done; the last one sums the row
// loss terms (block_sum_terms: double-float, a fixed order) over D, publishes n_valid and the
// error word, and resets the workspace header for the next call.  With local_counts,
// n_valid and n_bad (thread 0's) are this CTA's counts of the labels of its own rows,
// added to the header before the CTA counts itself done; the last CTA takes the totals.
template <int THREADS>
__device__ __forceinline__ void rows_finish(const CeRowParams& p, bool aborted, int n_valid, int n_bad,
                                            int* s_last, DFloat* dred, bool local_counts = false) {
    constexpr int WARPS = THREADS / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __syncthreads();
    unsigned e = 0;
    if (tid == 0) {
        if (local_counts) {
            if (n_valid) atomicAdd(&p.ws->nvalid, static_cast<unsigned>(n_valid));
            if (n_bad) atomicAdd(&p.ws->nbad, static_cast<unsigned>(n_bad));
        }
        if (aborted) atomicOr(&p.ws->err, static_cast<unsigned>(FOAK_ERRBIT_TIMEOUT));
        // The ticket releases this CTA's row terms, counts and error bits (the CTA
        // barrier above puts its other threads' writes before it) and, for the last
        // CTA, acquires everyone else's.
        const unsigned t = atom_add_acq_rel_gpu(&p.ws->done, 1u);
        const bool last = t == gridDim.x - 1;
        *s_last = last;
        if (last) {
            // Every other CTA has published its row terms and error bits and made its
            // last claim (the barrier below extends the acquire to the CTA's other
            // threads); the header is taken and reset now, its atomics' latency hidden
            // under the sum.
            e = atomicExch(&p.ws->err, 0u);
            if (local_counts) {
                n_valid = static_cast<int>(atomicExch(&p.ws->nvalid, 0u));
                n_bad = static_cast<int>(atomicExch(&p.ws->nbad, 0u));
            }
            atomicExch(&p.ws->next, 0u);
            atomicExch(&p.ws->done, 0u);
        }
    }
    __syncthreads();
    if (!*s_last) return;
    const DFloat tot = block_sum_terms<THREADS>(p.row_loss, p.N, dred);
    if (tid == 0) {
        *p.loss = df_div(tot, row_denominator(p, n_valid));
        if (p.n_valid) *p.n_valid = n_valid;
        if (n_bad > 0) e |= FOAK_ERRBIT_LABEL_RANGE;
        if (p.err) *p.err = static_cast<int32_t>(e);
    }
}

}  // namespace foak
