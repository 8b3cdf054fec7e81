// Row-wise cross-entropy: forward, and fused forward+backward in place.
//
// One row of the N x V logits matrix is owned by one CTA, or by a cluster of 2,
// 4 or 8 CTAs when the row is longer than one CTA's 64 KB slice (V = 128256 bf16
// needs 4, fp32 needs 8).  Each CTA stages its slice of the row in shared memory
// with one-dimensional bulk copies (TMA engine) completing on an mbarrier, keeps
// 2-4 rows in flight, and moves the slice into registers (8 x 16 bytes per
// thread).  From the registers it forms the thread's (max, sum exp(x - max)),
// merges the pairs across the warp (shuffles), the CTA (shared memory) and the
// cluster (distributed shared memory) into the row's log-sum-exp, and -- in the
// fused kernel -- writes (exp(x - lse) - onehot) * g / D straight from registers
// over the logits with 16-byte streaming stores.  Non-ignored rows are read
// once; ignored rows are never read (fused: only zero-filled).  That is the
// one-pass row sweep of the FastCrossEntropyLoss kernel the FOAK pages describe
// (fms-acceleration PR #79, Description item 4), re-planned for sm_103a.
//
// Rows whose address is not 16-byte aligned are split into a scalar head (< 16
// bytes), a run of 16-byte vectors and a scalar tail; the scalars are handled by
// one thread each.  n_valid is counted by every CTA from the labels (64 KB at
// N = 8192, an L2-resident read), and the mean loss is reduced in float64, in
// row order, by whichever CTA finishes last.
#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

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
constexpr size_t kSmemBudget = 227 * 1024 - 10 * 1024; // dynamic smem left after static use

struct CeRowParams {
    const char* x;
    char* dx;
    int64_t ld;
    const int64_t* labels;
    int64_t N, V, ignore_index;
    float g, denom;
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
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[16 / ES]) {
    if constexpr (ES == 2) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
}

template <int ES>
__device__ __forceinline__ uint4 pack(const float (&f)[16 / ES]) {
    uint4 v;
    if constexpr (ES == 2) {
        v.x = pack_bf16x2(f[0], f[1]);
        v.y = pack_bf16x2(f[2], f[3]);
        v.z = pack_bf16x2(f[4], f[5]);
        v.w = pack_bf16x2(f[6], f[7]);
    } else {
        v.x = __float_as_uint(f[0]); v.y = __float_as_uint(f[1]);
        v.z = __float_as_uint(f[2]); v.w = __float_as_uint(f[3]);
    }
    return v;
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

// Element e (runtime index) of a vector, without dynamic register indexing.
template <int ES>
__device__ __forceinline__ float vec_elem(const uint4& v, int e) {
    float f[16 / ES];
    unpack<ES>(v, f);
    float r = 0.f;
#pragma unroll
    for (int k = 0; k < 16 / ES; ++k)
        if (k == e) r = f[k];
    return r;
}

// The label's vector: same values as the fast path, minus scale at element e.
template <int ES>
__device__ __forceinline__ uint4 vec_grad_label(const uint4& v, int e_own, float c, bool mul, float scale) {
    constexpr int EPV = 16 / ES;
    float f[EPV], d[EPV];
    unpack<ES>(v, f);
#pragma unroll
    for (int k = 0; k < EPV; ++k) {
        float q = ex2(fmaf(f[k], kLog2e, -c));
        if (mul) q *= scale;
        d[k] = k == e_own ? q - scale : q;
    }
    return pack<ES>(d);
}

template <int ES, bool GRAD, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS == 256 ? 2 : 1) ce_rows_kernel(const CeRowParams p) {
    // slice: 512 x 8 or 1024 x 4 vectors (64 KB, one CTA per SM) or 256 x 8 (32 KB, two CTAs per SM)
    constexpr int VPT = THREADS == 256 ? 8 : kRowSliceVecMax / THREADS;
    constexpr int kRowThreads = THREADS;
    constexpr int kRowWarps = THREADS / 32;
    constexpr int EPV = 16 / ES;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bars[kRowMaxStages];
    __shared__ float2 red_ms[2][kRowWarps];
    __shared__ float2 xslot[2][kRowMaxCluster];  // [row parity][source CTA] (max, sum) pairs
    __shared__ uint64_t xbar[2];                  // completes when all K pairs of a row arrived
    __shared__ int64_t s_lab[kLabCache];
    __shared__ int iscratch[2 * kRowWarps];
    __shared__ double dred[kRowWarps];
    __shared__ int s_abort, s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.k;
    const int rank = K > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int64_t cid = K > 1 ? cluster_id_x() : blockIdx.x;
    const int64_t ncl = K > 1 ? cluster_count_x() : gridDim.x;
    const int64_t n_it = p.N > cid ? (p.N - 1 - cid) / ncl + 1 : 0;
    const int64_t row_bytes = p.ld * ES;
    const int tail_tid = K == 1 ? 32 : 0;
    const int64_t v0 = static_cast<int64_t>(rank) * p.per;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) mbar_init(&bars[s], 1);
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        fence_mbar_init();
        s_abort = 0;
        s_last = 0;
    }
    __syncthreads();
    if (K > 1) cluster_sync();  // every CTA's exchange barriers exist before the first st.async

    // Producer state (thread 0): next row iteration to look at, valid rows issued.
    int64_t p_it = 0;
    uint32_t p_v = 0;
    bool lab_cached = false;
    auto label_of = [&](int64_t it) -> int64_t {
        return (lab_cached && it < kLabCache) ? s_lab[it] : __ldg(p.labels + cid + it * ncl);
    };
    auto issue_next = [&]() {
        while (p_it < n_it) {
            const int64_t row = cid + p_it * ncl;
            const int64_t y = label_of(p_it);
            ++p_it;
            if (y == p.ignore_index || y < 0 || y >= p.V) continue;
            if (row == p.skip_load_row) {  // test hook: the stage's barrier is never completed
                ++p_v;
                return;
            }
            const char* rowp = p.x + row * row_bytes;
            const RowGeom gm = row_geom<ES>(rowp, p.V);
            int64_t nl = gm.nb - v0;
            nl = nl < 0 ? 0 : (nl > p.per ? p.per : nl);
            const uint32_t bytes = static_cast<uint32_t>(nl) * 16u;
            const int st = static_cast<int>(p_v % static_cast<uint32_t>(p.stages));
            ++p_v;
            uint64_t* bar = &bars[st];
            mbar_arrive_expect_tx(bar, bytes);
            const char* src = rowp + static_cast<int64_t>(gm.h) * ES + v0 * 16;
            unsigned char* dst = smem + static_cast<size_t>(st) * p.stage_bytes;
            for (uint32_t off = 0; off < bytes; off += kBulkChunk)
                bulk_g2s(dst + off, src + off, min(kBulkChunk, bytes - off), bar);
            return;
        }
    };
    if (tid == 0)
        for (int s = 0; s < p.stages; ++s) issue_next();

    int n_valid = 0, n_bad = 0;
    count_labels(p.count_labels, p.count_N, p.V, p.ignore_index, iscratch, n_valid, n_bad);
    const float D = p.denom > 0.f ? p.denom : static_cast<float>(n_valid);
    const float scale = p.g / D;
    // Labels of this CTA's first rows, for the row loop and the producer.
    for (int64_t it = tid; it < n_it && it < kLabCache; it += blockDim.x) s_lab[it] = __ldg(p.labels + cid + it * ncl);
    __syncthreads();
    lab_cached = true;

    // Gradient constants: for scale > 0 the scale is folded into the exponent,
    // 2^(x*log2e - lse2 + log2(scale)); otherwise the exponential is multiplied by it.
    const bool mul = !(scale > 0.f);
    const float log2_scale = mul ? 0.f : log2f(scale);

    int c_st = 0;          // stage of the next valid row
    uint32_t c_par = 0;    // its phase parity
    uint32_t c_v = 0;      // valid rows consumed
    bool aborted = false;
    for (int64_t it = 0; it < n_it; ++it) {
        const int64_t row = cid + it * ncl;
        const int64_t y = label_of(it);
        const bool valid = y != p.ignore_index && y >= 0 && y < p.V;
        const char* rowp = p.x + row * row_bytes;
        const RowGeom gm = row_geom<ES>(rowp, p.V);
        int nl;
        {
            const int64_t t = gm.nb - v0;
            nl = static_cast<int>(t < 0 ? 0 : (t > p.per ? p.per : t));
        }
        const bool has_head = rank == 0 && tid == 0 && gm.h > 0;
        const bool has_tail = rank == K - 1 && tid == tail_tid && gm.t > 0;
        const int64_t tail_col = gm.h + gm.nb * EPV;
        const int ns = has_head ? gm.h : (has_tail ? gm.t : 0);  // this thread's scalars
        const int64_t c0 = has_head ? 0 : tail_col;

        if (!valid) {
            if constexpr (GRAD) {
                char* drow = p.dx + row * row_bytes;
                uint4* dv = reinterpret_cast<uint4*>(drow + static_cast<int64_t>(gm.h) * ES + v0 * 16);
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                for (int i = tid; i < nl; i += kRowThreads) st_global_cs_v4(dv + i, z);
                for (int s = 0; s < ns; ++s) store_scalar<ES>(drow + (c0 + s) * ES, 0.f);
            }
            if (rank == 0 && tid == 0) {
                p.row_loss[row] = 0.f;
                if (p.lse) p.lse[row] = 0.f;
            }
            continue;
        }

        const int st = c_st;
        const uint32_t par = c_par;
        if (++c_st == p.stages) {
            c_st = 0;
            c_par ^= 1u;
        }
        ++c_v;
        if (!aborted && !mbar_wait_bounded(&bars[st], par, p.wait_ns)) s_abort = 1;

        // Slice -> registers (vectors past the slice hold -inf); scalars from global memory.
        uint4 v[VPT];
        const uint4* sb = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(st) * p.stage_bytes);
        const uint4 pad = RowMath<ES>::pad();
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int lv = tid + i * kRowThreads;
            v[i] = lv < nl ? sb[lv] : pad;
        }
        float xs[kMaxScalars];
        float m = RowMath<ES>::template vmax<VPT>(v);
        if (ns > 0) {
#pragma unroll
            for (int s = 0; s < kMaxScalars; ++s) {
                xs[s] = s < ns ? load_scalar<ES>(rowp + (c0 + s) * ES) : kNegInf;
                m = fmaxf(m, xs[s]);
            }
        }

        // Row (max, sum): the thread's sum is taken relative to its warp's max, the
        // warp's pair is published, and one barrier per row (which also frees the
        // stage for the producer) lets every warp merge the CTA's pairs.
        m = warp_max(m);
        const float mb = m == kNegInf ? 0.f : m * kLog2e;
        float sum = RowMath<ES>::template vsum<VPT>(v, mb);
        if (ns > 0) {
#pragma unroll
            for (int s = 0; s < kMaxScalars; ++s)
                if (s < ns) sum += ex2(fmaf(xs[s], kLog2e, -mb));
        }
        sum = warp_sum(sum);
        const int rb = c_v & 1;  // red[] is double-buffered by row parity
        if (lane == 0) red_ms[rb][warp] = make_float2(m, sum);
        __syncthreads();
        if (s_abort) aborted = true;
        if (tid == 0 && !aborted) {
            fence_proxy_async_smem();
            issue_next();
        }
        const float2 pr = lane < kRowWarps ? red_ms[rb][lane] : make_float2(kNegInf, 0.f);
        float M = warp_max(pr.x);
        float S = warp_sum(pr.x == kNegInf ? 0.f : pr.y * ex2((pr.x - M) * kLog2e));
        if (K > 1) {
            // cluster: thread 0 sends this CTA's pair to every CTA of the cluster with
            // st.async (no fence, so the row's gradient stores never have to drain
            // first); each CTA waits on its own barrier for the K pairs and merges them
            const uint32_t j = c_v - 1;
            const int xb = j & 1;
            if (tid == 0) {
                mbar_arrive_expect_tx(&xbar[xb], 8u * static_cast<uint32_t>(K));
                for (int r = 0; r < K; ++r)
                    st_async_f2(mapa_u32(&xslot[xb][rank], static_cast<uint32_t>(r)), M, S,
                                mapa_u32(&xbar[xb], static_cast<uint32_t>(r)));
            }
            if (!aborted && !mbar_wait_bounded(&xbar[xb], (j >> 1) & 1u, p.wait_ns)) s_abort = 1;
            const float2 q = lane < K ? xslot[xb][lane] : make_float2(kNegInf, 0.f);
            M = q.x;
            S = q.y;
            warp_ms_reduce(M, S);
            M = __shfl_sync(0xffffffffu, M, 0);
            S = __shfl_sync(0xffffffffu, S, 0);
        }
        const float lse2 = fmaf(M, kLog2e, lg2(S));  // log-sum-exp in base 2
        const float lse = lse2 * kLn2;

        // Which thread holds the label column (no division: kRowThreads is a power of 2).
        int own_slot = -1, own_e = 0, own_sc = -1;
        if (y < gm.h) {
            if (rank == 0 && tid == 0) own_sc = static_cast<int>(y);
        } else if (y < tail_col) {
            const int64_t ly = y - gm.h;
            const int64_t lv = ly / EPV - v0;
            if (lv >= 0 && lv < p.per && (static_cast<int>(lv) & (kRowThreads - 1)) == tid) {
                own_slot = static_cast<int>(lv) / kRowThreads;
                own_e = static_cast<int>(ly % EPV);
            }
        } else if (rank == K - 1 && tid == tail_tid) {
            own_sc = static_cast<int>(y - tail_col);
        }
        const bool owner = own_slot >= 0 || own_sc >= 0;
        if (owner) {
            float x_y = 0.f;
#pragma unroll
            for (int i = 0; i < VPT; ++i)
                if (i == own_slot) x_y = vec_elem<ES>(v[i], own_e);
#pragma unroll
            for (int s = 0; s < kMaxScalars; ++s)
                if (s == own_sc) x_y = xs[s];
            if (!aborted) p.row_loss[row] = lse - x_y;
        }

        if constexpr (GRAD) {
            const float c = lse2 - log2_scale;
            const f32x2_t L2 = f2_pack(kLog2e, kLog2e), C2 = f2_pack(-c, -c), S2 = f2_pack(scale, scale);
            char* drow = p.dx + row * row_bytes;
            uint4* dv = reinterpret_cast<uint4*>(drow + static_cast<int64_t>(gm.h) * ES + v0 * 16);
            if (!aborted) {
                if (!mul) {
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        const int lv = tid + i * kRowThreads;
                        uint4 o = RowMath<ES>::template vexp<false>(v[i], L2, C2, S2);
                        if (i == own_slot) o = vec_grad_label<ES>(v[i], own_e, c, false, scale);
                        if (lv < nl) st_global_cs_v4(dv + lv, o);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        const int lv = tid + i * kRowThreads;
                        uint4 o = RowMath<ES>::template vexp<true>(v[i], L2, C2, S2);
                        if (i == own_slot) o = vec_grad_label<ES>(v[i], own_e, c, true, scale);
                        if (lv < nl) st_global_cs_v4(dv + lv, o);
                    }
                }
                if (ns > 0) {
#pragma unroll
                    for (int s = 0; s < kMaxScalars; ++s) {
                        if (s < ns) {
                            float d = ex2(fmaf(xs[s], kLog2e, -c));
                            if (mul) d *= scale;
                            if (s == own_sc) d -= scale;
                            store_scalar<ES>(drow + (c0 + s) * ES, d);
                        }
                    }
                }
            }
        }
        if (rank == 0 && tid == 0 && p.lse && !aborted) p.lse[row] = lse;
    }

    // Loads still in flight exist only after an abort; let them land first.
    if (tid == 0) {
        while (c_v < p_v) {
            const int st = static_cast<int>(c_v % static_cast<uint32_t>(p.stages));
            (void)mbar_wait_bounded(&bars[st], (c_v / static_cast<uint32_t>(p.stages)) & 1u, p.wait_ns);
            ++c_v;
        }
    }
    if (K > 1) cluster_sync();  // no CTA leaves while a peer may still send it a pair

    __syncthreads();
    if (tid == 0) {
        if (aborted) atomicOr(&p.ws->err, static_cast<unsigned>(FOAK_ERRBIT_TIMEOUT));
        __threadfence();
        const unsigned t = atomicAdd(&p.ws->done, 1u);
        s_last = t == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;

    // Last CTA: loss = (sum of row terms in row order, float64) / D.
    __threadfence();
    double acc = 0.0;
    for (int64_t i = tid; i < p.N; i += kRowThreads) acc += static_cast<double>(__ldcg(p.row_loss + i));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, off);
    if (lane == 0) dred[warp] = acc;
    __syncthreads();
    if (tid == 0) {
        double tot = 0.0;
        for (int w = 0; w < kRowWarps; ++w) tot += dred[w];
        const double Dd = p.denom > 0.f ? static_cast<double>(p.denom) : static_cast<double>(n_valid);
        *p.loss = static_cast<float>(tot / Dd);
        if (p.n_valid) *p.n_valid = n_valid;
        unsigned e = atomicExch(&p.ws->err, 0u);
        if (n_bad > 0) e |= FOAK_ERRBIT_LABEL_RANGE;
        if (p.err) *p.err = static_cast<int32_t>(e);
        atomicExch(&p.ws->done, 0u);
    }
}

// ------------------------------------------------------------------ host side

int64_t ce_rows_max_vocab(int elem_bytes) {
    return static_cast<int64_t>(kRowMaxCluster) * kRowSliceVecMax * (16 / elem_bytes);
}

namespace {

struct Plan {
    int threads, k, per, stages;
    uint32_t stage_bytes;
    size_t smem;
};

constexpr size_t kSmemBudgetHalf = 100 * 1024;  // per CTA when two CTAs share an SM

// Smallest cluster whose per-CTA slices fit `slice_max` vectors.
bool plan_with(int ES, int64_t V, int threads, int64_t slice_max, size_t budget, Plan* pl) {
    const int64_t nb_max = V * ES / 16;
    for (int k = 1; k <= kRowMaxCluster; k *= 2) {
        const int64_t per = (nb_max + k - 1) / k;
        if (per <= slice_max) {
            pl->threads = threads;
            pl->k = k;
            pl->per = static_cast<int>(std::max<int64_t>(per, 1));
            pl->stage_bytes = static_cast<uint32_t>(((pl->per * 16 + 127) / 128) * 128);
            pl->stages = static_cast<int>(std::min<size_t>(kRowMaxStages, budget / pl->stage_bytes));
            pl->smem = static_cast<size_t>(pl->stages) * pl->stage_bytes;
            return pl->stages >= 2;
        }
    }
    return false;
}

// Rows that fit one 64 KB slice: one 512-thread CTA per row and SM.  Longer rows
// need a cluster anyway; there 32 KB slices on 256-thread CTAs, two per SM, hide
// each other's per-row latency better (when eight of them cover the row).
bool plan_rows(int ES, int64_t V, Plan* pl) {
    static const int forced = [] {
        const char* e = std::getenv("FOAK_ROW_THREADS");  // tuning override: 256, 512 or 1024
        return e ? std::atoi(e) : 0;
    }();
    if (forced == 1024 && plan_with(ES, V, 1024, kRowSliceVecMax, kSmemBudget, pl)) return true;
    if (forced == 256 && plan_with(ES, V, 256, 2048, kSmemBudgetHalf, pl)) return true;
    if (!plan_with(ES, V, 512, kRowSliceVecMax, kSmemBudget, pl)) return false;
    if (forced == 0 && pl->k > 1) {
        Plan half;
        if (plan_with(ES, V, 256, 2048, kSmemBudgetHalf, &half)) *pl = half;
    }
    return true;
}

std::mutex g_mu;
std::map<std::tuple<int, const void*, int, size_t>, int> g_clusters;  // (device, kernel, k, smem)
std::map<std::pair<int, const void*>, bool> g_attr_set;                // (device, kernel)

// Co-resident clusters for this kernel configuration (cached per device).  The
// kernel's dynamic shared-memory limit is raised once per device to the full
// budget, so every plan's size fits whatever order plans are launched in.
cudaError_t resident_clusters(const void* kern, int threads, int k, size_t smem, int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    auto key = std::make_tuple(dev, kern, k, smem);
    auto it = g_clusters.find(key);
    if (it != g_clusters.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    auto akey = std::make_pair(dev, kern);
    if (!g_attr_set[akey]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBudget));
        if (e != cudaSuccess) return e;
        g_attr_set[akey] = true;
    }
    int n = 0;
    if (k == 1) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
        if (e != cudaSuccess) return e;
        n = per_sm * device_sm_count();
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(k), 1, 1);
        cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(k);
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
    }
    if (n < 1) n = 1;
    g_clusters[key] = n;
    *out = n;
    return cudaSuccess;
}

template <int ES, bool GRAD, int THREADS>
cudaError_t launch_typed(const CeRowParams& base, const Plan& pl, cudaStream_t stream) {
    const void* kern = reinterpret_cast<const void*>(&ce_rows_kernel<ES, GRAD, THREADS>);
    int ncl = 0;
    cudaError_t e = resident_clusters(kern, THREADS, pl.k, pl.smem, &ncl);
    if (e != cudaSuccess) return e;
    const int64_t want = std::max<int64_t>(1, std::min<int64_t>(ncl, base.N));
    CeRowParams prm = base;
    prm.k = pl.k;
    prm.per = pl.per;
    prm.stages = pl.stages;
    prm.stage_bytes = pl.stage_bytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want * pl.k), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(pl.k);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ce_rows_kernel<ES, GRAD, THREADS>, prm);
}

template <int ES, bool GRAD>
cudaError_t launch_vpt(const CeRowParams& base, const Plan& pl, cudaStream_t stream) {
    if (pl.threads == 256) return launch_typed<ES, GRAD, 256>(base, pl, stream);
    return pl.threads == 1024 ? launch_typed<ES, GRAD, 1024>(base, pl, stream)
                              : launch_typed<ES, GRAD, 512>(base, pl, stream);
}

}  // namespace

cudaError_t launch_ce_rows(bool grad, int elem_bytes, const void* x, void* dx, int64_t ld,
                           const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index, float g,
                           float denom, float* loss, float* lse, float* row_loss, int32_t* n_valid,
                           int32_t* err, CeWsHeader* ws, cudaStream_t stream, const int64_t* count_labels,
                           int64_t count_N) {
    Plan pl;
    if (!plan_rows(elem_bytes, V, &pl)) return cudaErrorInvalidValue;
    CeRowParams prm = {};
    prm.x = static_cast<const char*>(x);
    prm.dx = static_cast<char*>(dx);
    prm.ld = ld;
    prm.labels = labels;
    prm.N = N;
    prm.V = V;
    prm.ignore_index = ignore_index;
    prm.g = g;
    prm.denom = denom;
    prm.loss = loss;
    prm.lse = lse;
    prm.row_loss = row_loss;
    prm.n_valid = n_valid;
    prm.err = err;
    prm.ws = ws;
    prm.count_labels = count_labels ? count_labels : labels;
    prm.count_N = count_labels ? count_N : N;
    prm.wait_ns = test_wait_limit_ns();
    prm.skip_load_row = test_skip_load_row();
    if (elem_bytes == 2)
        return grad ? launch_vpt<2, true>(prm, pl, stream) : launch_vpt<2, false>(prm, pl, stream);
    return grad ? launch_vpt<4, true>(prm, pl, stream) : launch_vpt<4, false>(prm, pl, stream);
}

}  // namespace foak
