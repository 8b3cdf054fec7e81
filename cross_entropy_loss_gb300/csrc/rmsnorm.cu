// RMSNorm forward and backward -- the "Fast RMS LayerNorm" kernels the FOAK pages
// list among their fused operations (fms-acceleration-foak 0.7.4 page; the patch
// rule there swaps a decoder's RMSNorm module for fast_rms_layernorm).  The pages
// print no formula; the operation is the decoders' RMSNorm:
//     r_i = 1 / sqrt(mean_j x_ij^2 + eps),   y_ij = x_ij * r_i * gamma_j
// computed in fp32 and rounded once to the storage type, and its gradients
//     xh = x * r,  u = gamma * dy,  dx = r * (u - xh * mean(xh * u)),
//     dgamma_j = sum_i dy_ij * xh_ij.
//
// Both row kernels give one warp a row (D elements, 16-byte vectors, D % 8 == 0)
// and read it twice: the first pass reduces over the row, the second re-reads it
// (from L1: 8 KB at D = 4096 bf16) and writes.  HBM traffic is the algorithmic
// one: forward reads X and writes Y; backward reads dY and X and writes dX.  dgamma
// is a column reduction over rows: a separate kernel gives each thread 8
// consecutive columns and one of 128 row groups, writes per-group partials, and a
// last kernel sums the 128 partials in a fixed order -- deterministic, no atomics.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "foak_ce.h"
#include "internal.h"

namespace foak {

namespace {

constexpr int kNormThreads = 256;  // 8 warps, one row each at a time
constexpr int kGammaThreads = 128;

template <int ES>
__device__ __forceinline__ void load8(const char* p, float (&f)[16 / ES]) {
    const uint4 v = ld_global_v4(reinterpret_cast<const uint4*>(p));
    if constexpr (ES == 2) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
}

template <int ES>
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[16 / ES]) {
    if constexpr (ES == 2) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
}

__device__ __forceinline__ uint4 ldv(const char* p) { return ld_global_v4(reinterpret_cast<const uint4*>(p)); }

// The loops below take four 16-byte vectors (or rows) at a time and issue all of their
// loads before any arithmetic: the loads are ordered asm, so arithmetic placed between
// them would cost a round trip per vector.  The arithmetic keeps the one-at-a-time order.
constexpr int kBatch = 4;

template <int ES>
__device__ __forceinline__ void store8(char* p, const float (&f)[16 / ES]) {
    uint4 v;
    if constexpr (ES == 2) {
        v.x = pack_bf16x2(f[0], f[1]); v.y = pack_bf16x2(f[2], f[3]);
        v.z = pack_bf16x2(f[4], f[5]); v.w = pack_bf16x2(f[6], f[7]);
    } else {
        v.x = __float_as_uint(f[0]); v.y = __float_as_uint(f[1]);
        v.z = __float_as_uint(f[2]); v.w = __float_as_uint(f[3]);
    }
    *reinterpret_cast<uint4*>(p) = v;
}

template <int ES>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_fwd_kernel(const char* __restrict__ X, int64_t ldx,
                                                                   const char* __restrict__ gamma, int64_t N,
                                                                   int64_t D, float eps, char* __restrict__ Y,
                                                                   int64_t ldy, float* __restrict__ rstd) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    constexpr int EPV = 16 / ES;
    const int lane = threadIdx.x & 31;
    const int64_t nvec = D / EPV;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kNormThreads / 32);
    for (int64_t row = blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5); row < N; row += warps) {
        const char* x = X + row * ldx * ES;
        float ss = 0.f;
        for (int64_t v0 = lane; v0 < nvec; v0 += kBatch * 32) {
            uint4 w[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (v0 + 32 * u < nvec) w[u] = ldv(x + (v0 + 32 * u) * 16);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (v0 + 32 * u < nvec) {
                    float f[EPV];
                    unpack<ES>(w[u], f);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) ss = fmaf(f[k], f[k], ss);
                }
            }
        }
        ss = warp_sum(ss);
        const float r = rsqrtf(ss / static_cast<float>(D) + eps);
        char* y = Y + row * ldy * ES;
        for (int64_t v0 = lane; v0 < nvec; v0 += kBatch * 32) {
            uint4 w[kBatch], gw[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (v0 + 32 * u < nvec) {
                    w[u] = ldv(x + (v0 + 32 * u) * 16);
                    gw[u] = ldv(gamma + (v0 + 32 * u) * 16);
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (v0 + 32 * u < nvec) {
                    float f[EPV], gm[EPV];
                    unpack<ES>(w[u], f);
                    unpack<ES>(gw[u], gm);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) f[k] = f[k] * r * gm[k];
                    store8<ES>(y + (v0 + 32 * u) * 16, f);
                }
            }
        }
        if (lane == 0 && rstd) rstd[row] = r;
    }
}

// Rows of at most 32 * VPL vectors: the warp holds its row in registers (lane l has
// vectors l, l + 32, ...), so every load of the row is in flight at once and the row
// is read from memory once; same arithmetic, in the same order, as rmsnorm_fwd_kernel.
template <int ES, int VPL>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_fwd_reg_kernel(const char* __restrict__ X, int64_t ldx,
                                                                       const char* __restrict__ gamma, int64_t N,
                                                                       int64_t D, float eps, char* __restrict__ Y,
                                                                       int64_t ldy, float* __restrict__ rstd) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    constexpr int EPV = 16 / ES;
    const int lane = threadIdx.x & 31;
    const int nvec = static_cast<int>(D / EPV);
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kNormThreads / 32);
    for (int64_t row = blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5); row < N; row += warps) {
        const uint4* x = reinterpret_cast<const uint4*>(X + row * ldx * ES);
        uint4 v[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int j = lane + 32 * i;
            v[i] = j < nvec ? ld_global_v4(x + j) : make_uint4(0u, 0u, 0u, 0u);
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (lane + 32 * i < nvec) {
                float f[EPV];
                unpack<ES>(v[i], f);
#pragma unroll
                for (int k = 0; k < EPV; ++k) ss = fmaf(f[k], f[k], ss);
            }
        }
        ss = warp_sum(ss);
        const float r = rsqrtf(ss / static_cast<float>(D) + eps);
        char* y = Y + row * ldy * ES;
#pragma unroll
        for (int i0 = 0; i0 < VPL; i0 += kBatch) {  // gamma's loads (L1) a batch at a time
            uint4 gw[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (i0 + u < VPL && lane + 32 * (i0 + u) < nvec) gw[u] = ldv(gamma + static_cast<int64_t>(lane + 32 * (i0 + u)) * 16);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = i0 + u;
                const int j = lane + 32 * i;
                if (i < VPL && j < nvec) {
                    float f[EPV], gm[EPV];
                    unpack<ES>(v[i], f);
                    unpack<ES>(gw[u], gm);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) f[k] = f[k] * r * gm[k];
                    store8<ES>(y + static_cast<int64_t>(j) * 16, f);
                }
            }
        }
        if (lane == 0 && rstd) rstd[row] = r;
    }
}

template <int ES>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_bwd_kernel(const char* __restrict__ dY, int64_t lddy,
                                                                   const char* __restrict__ X, int64_t ldx,
                                                                   const char* __restrict__ gamma,
                                                                   const float* __restrict__ rstd, int64_t N,
                                                                   int64_t D, char* __restrict__ dX, int64_t lddx) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    constexpr int EPV = 16 / ES;
    const int lane = threadIdx.x & 31;
    const int64_t nvec = D / EPV;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kNormThreads / 32);
    for (int64_t row = blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5); row < N; row += warps) {
        const char* x = X + row * ldx * ES;
        const char* dy = dY + row * lddy * ES;
        const float r = rstd[row];
        float dot = 0.f;  // sum of xh * u over the row
        for (int64_t v0 = lane; v0 < nvec; v0 += kBatch * 32) {
            uint4 wx[kBatch], wd[kBatch], wg[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t v = v0 + 32 * u;
                if (v < nvec) {
                    wx[u] = ldv(x + v * 16);
                    wd[u] = ldv(dy + v * 16);
                    wg[u] = ldv(gamma + v * 16);
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (v0 + 32 * u < nvec) {
                    float fx[EPV], fd[EPV], gm[EPV];
                    unpack<ES>(wx[u], fx);
                    unpack<ES>(wd[u], fd);
                    unpack<ES>(wg[u], gm);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) dot = fmaf(fx[k] * r, gm[k] * fd[k], dot);
                }
            }
        }
        dot = warp_sum(dot);
        const float m = dot / static_cast<float>(D);
        char* dx = dX + row * lddx * ES;
        for (int64_t v0 = lane; v0 < nvec; v0 += kBatch * 32) {
            uint4 wx[kBatch], wd[kBatch], wg[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t v = v0 + 32 * u;
                if (v < nvec) {
                    wx[u] = ldv(x + v * 16);
                    wd[u] = ldv(dy + v * 16);
                    wg[u] = ldv(gamma + v * 16);
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t v = v0 + 32 * u;
                if (v < nvec) {
                    float fx[EPV], fd[EPV], gm[EPV], o[EPV];
                    unpack<ES>(wx[u], fx);
                    unpack<ES>(wd[u], fd);
                    unpack<ES>(wg[u], gm);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) o[k] = r * (gm[k] * fd[k] - fx[k] * r * m);
                    store8<ES>(dx + v * 16, o);
                }
            }
        }
    }
}

// part[g][j] = sum over rows i = g, g + G, ... of dy_ij * x_ij * r_i; thread = 8 columns.
template <int ES>
__global__ void __launch_bounds__(kGammaThreads) rmsnorm_dgamma_kernel(const char* __restrict__ dY, int64_t lddy,
                                                                       const char* __restrict__ X, int64_t ldx,
                                                                       const float* __restrict__ rstd, int64_t N,
                                                                       int64_t D, float* __restrict__ part) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    constexpr int EPV = 16 / ES;
    const int64_t v = static_cast<int64_t>(blockIdx.x) * kGammaThreads + threadIdx.x;  // vector of columns
    if (v * EPV >= D) return;
    const int64_t grp = blockIdx.y, G = gridDim.y;
    float acc[EPV];
#pragma unroll
    for (int k = 0; k < EPV; ++k) acc[k] = 0.f;
    for (int64_t i0 = grp; i0 < N; i0 += kBatch * G) {
        uint4 wx[kBatch], wd[kBatch];
        float r[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int64_t i = i0 + u * G;
            if (i < N) {
                wx[u] = ldv(X + (i * ldx + v * EPV) * ES);
                wd[u] = ldv(dY + (i * lddy + v * EPV) * ES);
                r[u] = rstd[i];
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (i0 + u * G < N) {
                float fx[EPV], fd[EPV];
                unpack<ES>(wx[u], fx);
                unpack<ES>(wd[u], fd);
#pragma unroll
                for (int k = 0; k < EPV; ++k) acc[k] = fmaf(fd[k], fx[k] * r[u], acc[k]);
            }
        }
    }
    float* p = part + grp * D + v * EPV;
#pragma unroll
    for (int k = 0; k < EPV; ++k) p[k] = acc[k];
}

// At most this many CTAs write dgamma partials (the workspace holds 512 x D floats).
constexpr int kPartMaxGrid = 512;

// 16-byte copy global -> shared by this thread, completed by its own wait_group
// (a hardware wait, no spin): the pre-bulk asynchronous copy, used here because every
// thread reads back exactly the vectors it copied.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int PENDING>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
}

// The one-pass backward with the rows streamed through a shared-memory ring: thread v
// owns column vectors v, v + threads, ... (VPT of them), each CTA takes one contiguous
// range of rows in batches of RR, and every thread copies its own vectors of X and dY
// for the batch kRingStages - 1 ahead of the one it works on, so copies stay in flight
// through each batch's reduction barrier.  Per row, with u = gamma * dY and s = sum_j x_j u_j:
//     m = r s / D,   dX = r u - (r m) (x r),   dgamma += dY (x r)
// (r factored out of the row sum), on element pairs with the two-wide FP32
// instructions (each half rounded as the scalar operation): the kernel is bound by
// instruction issue before it is by memory.
constexpr int kRingStages = 3;
constexpr int kRingSmemMax = 220 * 1024;
constexpr int kRingRows = 2;        // rows per batch (one barrier each)
constexpr int kRingVpt = 2;         // 16-byte column vectors per thread, rows of <= 512 vectors
constexpr int kRingVptWide = 4;     // the same for rows of 513 to 1024 vectors
constexpr int kRingMaxThreads = 256;  // rows of up to 8192 bf16 / 4096 fp32 elements
// two CTAs per SM at 4096 bf16 (96 KB of ring each), one for the wide rows (192 KB)
constexpr int ring_min_blocks(int vpt) { return vpt <= 2 ? 2 : 1; }

__host__ __device__ constexpr size_t ring_stage_bytes(int rows, int vpt, int threads) {
    return static_cast<size_t>(rows) * 2 * vpt * static_cast<size_t>(threads) * 16;
}
static_assert(kRingStages * ring_stage_bytes(kRingRows, kRingVptWide, kRingMaxThreads) <=
                  static_cast<size_t>(kRingSmemMax),
              "ring too large");

// A 16-byte vector as element pairs, and back (bf16 rounded to nearest even).
template <int ES>
__device__ __forceinline__ void unpack_pairs(const uint4& w, float2 (&p)[8 / ES]) {
    if constexpr (ES == 2) {
        p[0] = make_float2(bf16_lo(w.x), bf16_hi(w.x));
        p[1] = make_float2(bf16_lo(w.y), bf16_hi(w.y));
        p[2] = make_float2(bf16_lo(w.z), bf16_hi(w.z));
        p[3] = make_float2(bf16_lo(w.w), bf16_hi(w.w));
    } else {
        p[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
        p[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
}

template <int ES>
__device__ __forceinline__ void store_pairs(char* dst, const float2 (&p)[8 / ES]) {
    uint4 w;
    if constexpr (ES == 2) {
        w = make_uint4(pack_bf16x2(p[0].x, p[0].y), pack_bf16x2(p[1].x, p[1].y), pack_bf16x2(p[2].x, p[2].y),
                       pack_bf16x2(p[3].x, p[3].y));
    } else {
        w = make_uint4(__float_as_uint(p[0].x), __float_as_uint(p[0].y), __float_as_uint(p[1].x),
                       __float_as_uint(p[1].y));
    }
    *reinterpret_cast<uint4*>(dst) = w;
}

// DG: dgamma wanted (the partials are written); without it part is not touched.
template <int ES, int RR, int VPT, bool DG>
__global__ void __launch_bounds__(kRingMaxThreads, ring_min_blocks(VPT))
    rmsnorm_bwd_ring_kernel(const char* __restrict__ dY, int64_t lddy, const char* __restrict__ X, int64_t ldx,
                            const char* __restrict__ gamma, const float* __restrict__ rstd, int64_t N, int64_t D,
                            char* __restrict__ dX, int64_t lddx, float* __restrict__ part) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    constexpr int EPV = 16 / ES, NP = EPV / 2;
    extern __shared__ uint4 ring[];  // [kRingStages][RR][X, dY][VPT][threads]
    __shared__ float red[2][RR][32];
    const int v = threadIdx.x, lane = v & 31, warp = v >> 5, nt = blockDim.x, warps = nt >> 5;
    bool act[VPT];  // thread v owns column vectors v, v + nt, ...
#pragma unroll
    for (int j = 0; j < VPT; ++j) act[j] = static_cast<int64_t>(v + j * nt) * EPV < D;
    const int64_t G = gridDim.x;
    const int64_t r_begin = N * static_cast<int64_t>(blockIdx.x) / G;
    const int64_t r_end = N * (static_cast<int64_t>(blockIdx.x) + 1) / G;
    const int64_t nb = (r_end - r_begin + RR - 1) / RR;
    const float inv_d = 1.f / static_cast<float>(D);
    // batch b's copies into slot b % kRingStages, one commit group per batch (empty
    // past the last batch, so that the group count stays in step)
    auto issue = [&](int64_t b) {
        if (b < nb) {
            uint4* slot = ring + static_cast<size_t>(b % kRingStages) * (RR * 2 * VPT) * nt;
#pragma unroll
            for (int q = 0; q < RR; ++q) {
                const int64_t row = r_begin + b * RR + q;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (row < r_end && act[j]) {
                        const int64_t col = static_cast<int64_t>(v + j * nt) * EPV;
                        cp_async16(slot + ((2 * q) * VPT + j) * nt + v, X + (row * ldx + col) * ES);
                        cp_async16(slot + ((2 * q + 1) * VPT + j) * nt + v, dY + (row * lddy + col) * ES);
                    }
                }
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < kRingStages - 1; ++s) issue(s);
    float2 gm2[VPT][NP], acc2[VPT][NP];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        unpack_pairs<ES>(act[j] ? ldv(gamma + static_cast<int64_t>(v + j * nt) * 16) : make_uint4(0u, 0u, 0u, 0u),
                         gm2[j]);
#pragma unroll
        for (int k = 0; k < NP; ++k) acc2[j][k] = make_float2(0.f, 0.f);
    }
    float rn[RR];
#pragma unroll
    for (int q = 0; q < RR; ++q) rn[q] = r_begin + q < r_end ? rstd[r_begin + q] : 0.f;
    int par = 0;
    for (int64_t b = 0; b < nb; ++b, par ^= 1) {
        // the slot of batch b - 1, read before the last barrier, takes batch b + kRingStages - 1
        issue(b + kRingStages - 1);
        const int64_t row0 = r_begin + b * RR;
        float r[RR];
#pragma unroll
        for (int q = 0; q < RR; ++q) {
            r[q] = rn[q];
            const int64_t nxt = row0 + RR + q;
            rn[q] = nxt < r_end ? rstd[nxt] : 0.f;
        }
        cp_async_wait<kRingStages - 1>();  // this thread's copies of batch b have landed
        const uint4* slot = ring + static_cast<size_t>(b % kRingStages) * (RR * 2 * VPT) * nt;
        // the batch is read from the ring twice, before and after the barrier (nothing
        // held through it; the slot is refilled only in the next iteration)
#pragma unroll
        for (int q = 0; q < RR; ++q) {
            float2 d2 = make_float2(0.f, 0.f);
            if (row0 + q < r_end) {
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (act[j]) {
                        float2 x[NP], d[NP];
                        unpack_pairs<ES>(slot[((2 * q) * VPT + j) * nt + v], x);
                        unpack_pairs<ES>(slot[((2 * q + 1) * VPT + j) * nt + v], d);
#pragma unroll
                        for (int k = 0; k < NP; ++k) d2 = __ffma2_rn(x[k], __fmul2_rn(gm2[j][k], d[k]), d2);
                    }
                }
            }
            const float dot = warp_sum(d2.x + d2.y);
            if (lane == 0) red[par][q][warp] = dot;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < RR; ++q) {
            const int64_t row = row0 + q;
            const float s = warp_sum(lane < warps ? red[par][q][lane] : 0.f);
            if (row < r_end) {
                const float rm = r[q] * (r[q] * s * inv_d);
                const float2 r2 = make_float2(r[q], r[q]), nrm2 = make_float2(-rm, -rm);
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (act[j]) {
                        float2 x[NP], d[NP], o[NP];
                        unpack_pairs<ES>(slot[((2 * q) * VPT + j) * nt + v], x);
                        unpack_pairs<ES>(slot[((2 * q + 1) * VPT + j) * nt + v], d);
#pragma unroll
                        for (int k = 0; k < NP; ++k) {
                            const float2 xh = __fmul2_rn(x[k], r2);
                            o[k] = __ffma2_rn(nrm2, xh, __fmul2_rn(r2, __fmul2_rn(gm2[j][k], d[k])));
                            if constexpr (DG) acc2[j][k] = __ffma2_rn(d[k], xh, acc2[j][k]);
                        }
                        store_pairs<ES>(dX + (row * lddx + static_cast<int64_t>(v + j * nt) * EPV) * ES, o);
                    }
                }
            }
        }
    }
    cp_async_wait<0>();  // no copy outlives the CTA (the trailing groups are empty)
    if constexpr (DG) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (act[j]) {
                float* p = part + static_cast<int64_t>(blockIdx.x) * D + static_cast<int64_t>(v + j * nt) * EPV;
#pragma unroll
                for (int k = 0; k < NP; ++k) {
                    p[2 * k] = acc2[j][k].x;
                    p[2 * k + 1] = acc2[j][k].y;
                }
            }
        }
    }
}

// The forward through the same kind of ring, for rows too wide for one warp's
// registers: thread v owns column vectors v, v + threads, ... (VPT of them) of every
// row, each CTA takes one contiguous range of rows in batches of RR, and every thread
// copies its own vectors of X kRingStages - 1 batches ahead.  Per row the CTA sums
// x^2 (pairs on the two-wide FP32 instructions, then warp shuffles and one barrier per
// batch), and each thread writes y = x r gamma for its vectors (x r rounded, then times
// gamma, as the other forward kernels).
template <int ES, int RR, int VPT>
__global__ void __launch_bounds__(kRingMaxThreads, 2)
    rmsnorm_fwd_cta_ring_kernel(const char* __restrict__ X, int64_t ldx, const char* __restrict__ gamma, int64_t N,
                                int64_t D, float eps, char* __restrict__ Y, int64_t ldy, float* __restrict__ rstd) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    constexpr int EPV = 16 / ES, NP = EPV / 2;
    extern __shared__ uint4 ring[];  // [kRingStages][RR][VPT][threads]
    __shared__ float red[2][RR][32];
    const int v = threadIdx.x, lane = v & 31, warp = v >> 5, nt = blockDim.x, warps = nt >> 5;
    bool act[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) act[j] = static_cast<int64_t>(v + j * nt) * EPV < D;
    const int64_t G = gridDim.x;
    const int64_t r_begin = N * static_cast<int64_t>(blockIdx.x) / G;
    const int64_t r_end = N * (static_cast<int64_t>(blockIdx.x) + 1) / G;
    const int64_t nb = (r_end - r_begin + RR - 1) / RR;
    auto issue = [&](int64_t b) {  // one commit group per batch (empty past the last)
        if (b < nb) {
            uint4* slot = ring + static_cast<size_t>(b % kRingStages) * (RR * VPT) * nt;
#pragma unroll
            for (int q = 0; q < RR; ++q) {
                const int64_t row = r_begin + b * RR + q;
#pragma unroll
                for (int j = 0; j < VPT; ++j)
                    if (row < r_end && act[j])
                        cp_async16(slot + (q * VPT + j) * nt + v,
                                   X + (row * ldx + static_cast<int64_t>(v + j * nt) * EPV) * ES);
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int s = 0; s < kRingStages - 1; ++s) issue(s);
    float2 gm2[VPT][NP];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
        unpack_pairs<ES>(act[j] ? ldv(gamma + static_cast<int64_t>(v + j * nt) * 16) : make_uint4(0u, 0u, 0u, 0u),
                         gm2[j]);
    int par = 0;
    for (int64_t b = 0; b < nb; ++b, par ^= 1) {
        issue(b + kRingStages - 1);  // into the slot read before the last barrier
        cp_async_wait<kRingStages - 1>();
        const int64_t row0 = r_begin + b * RR;
        const uint4* slot = ring + static_cast<size_t>(b % kRingStages) * (RR * VPT) * nt;
#pragma unroll
        for (int q = 0; q < RR; ++q) {
            float2 s2 = make_float2(0.f, 0.f);
            if (row0 + q < r_end) {
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (act[j]) {
                        float2 x[NP];
                        unpack_pairs<ES>(slot[(q * VPT + j) * nt + v], x);
#pragma unroll
                        for (int k = 0; k < NP; ++k) s2 = __ffma2_rn(x[k], x[k], s2);
                    }
                }
            }
            const float ss = warp_sum(s2.x + s2.y);
            if (lane == 0) red[par][q][warp] = ss;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < RR; ++q) {
            const int64_t row = row0 + q;
            const float ss = warp_sum(lane < warps ? red[par][q][lane] : 0.f);
            if (row < r_end) {
                const float r = rsqrtf(ss / static_cast<float>(D) + eps);
                const float2 r2 = make_float2(r, r);
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (act[j]) {
                        float2 x[NP];
                        unpack_pairs<ES>(slot[(q * VPT + j) * nt + v], x);
#pragma unroll
                        for (int k = 0; k < NP; ++k) x[k] = __fmul2_rn(__fmul2_rn(x[k], r2), gm2[j][k]);
                        store_pairs<ES>(Y + (row * ldy + static_cast<int64_t>(v + j * nt) * EPV) * ES, x);
                    }
                }
                if (v == 0 && rstd) rstd[row] = r;
            }
        }
    }
    cp_async_wait<0>();  // no copy outlives the CTA (the trailing groups are empty)
}

// dgamma[j] = sum of part[g][j] over g < G (G <= kRedMaxG for every caller), in a
// fixed order: 32 slices of 32 columns per CTA, slice sl loading g = sl, sl + 32, ...
// all at once (one round trip) and adding them in g order, then slice 0 adding the 32
// slice sums in slice order.  (Four running sums fed four loads at a time took
// 4.9 us for 304 partials of 4096; 8 slices of 64 columns took 7.8 us.)
constexpr int kRedCols = 32, kRedSlices = 32, kRedMaxG = 512;
static_assert(kPartMaxGrid <= kRedMaxG && kRmsGammaGroups <= kRedMaxG, "partials beyond the reduce's reach");
__global__ void __launch_bounds__(kRedCols * kRedSlices) rmsnorm_dgamma_reduce(const float* __restrict__ part, int G,
                                                                             int64_t D, float* __restrict__ dgamma) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    __shared__ float ss[kRedSlices][kRedCols];
    const int c = threadIdx.x % kRedCols, sl = threadIdx.x / kRedCols;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kRedCols + c;
    float s = 0.f;
    if (j < D) {
        float val[kRedMaxG / kRedSlices];
#pragma unroll
        for (int i = 0; i < kRedMaxG / kRedSlices; ++i) {
            const int g = sl + i * kRedSlices;
            val[i] = g < G ? part[static_cast<int64_t>(g) * D + j] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kRedMaxG / kRedSlices; ++i) s += val[i];
    }
    ss[sl][c] = s;
    __syncthreads();
    if (sl == 0 && j < D) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < kRedSlices; ++k) t += ss[k][c];
        dgamma[j] = t;
    }
}

int norm_grid(int64_t N) {
    const int64_t rows_per_cta = kNormThreads / 32;
    const int64_t want = (N + rows_per_cta - 1) / rows_per_cta;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(device_sm_count()) * 8)));
}

std::mutex g_ring_mu;
bool g_ring_attr[64][8] = {};

// The ring kernel's shared memory limit, set once per device, element size and width.
template <int ES, int VPT, bool DG>
cudaError_t ring_attr() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int k = (ES == 2 ? 0 : 4) + (VPT == kRingVpt ? 0 : 2) + (DG ? 0 : 1);
    std::lock_guard<std::mutex> lock(g_ring_mu);
    if (!g_ring_attr[dev][k]) {
        e = cudaFuncSetAttribute(rmsnorm_bwd_ring_kernel<ES, kRingRows, VPT, DG>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemMax);
        if (e != cudaSuccess) return e;
        g_ring_attr[dev][k] = true;
    }
    return cudaSuccess;
}

// The one-pass backward through the shared-memory ring: as many CTAs per SM as its
// shared memory and threads allow, each with a contiguous range of rows; then the
// fixed-order dgamma reduce over the CTAs' partials.
template <int ES, int VPT, bool DG>
cudaError_t launch_bwd_ring(const char* dy, int64_t lddy, const char* x, int64_t ldx, const char* g, const float* rstd,
                            int64_t N, int64_t D, char* dx, int64_t lddx, float* part, float* dgamma, cudaStream_t s) {
    const int64_t nvec = D / (16 / ES);
    const int threads = static_cast<int>(((nvec + VPT - 1) / VPT + 31) / 32 * 32);
    const size_t smem = kRingStages * ring_stage_bytes(kRingRows, VPT, threads);
    cudaError_t e = ring_attr<ES, VPT, DG>();
    if (e != cudaSuccess) return e;
    int per_sm = 0;  // every CTA resident at once: the row ranges are contiguous
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rmsnorm_bwd_ring_kernel<ES, kRingRows, VPT, DG>, threads,
                                                      smem);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(std::min<int64_t>(
        {N, static_cast<int64_t>(device_sm_count()) * std::max(per_sm, 1), kPartMaxGrid}));
    e = launch_dependent(rmsnorm_bwd_ring_kernel<ES, kRingRows, VPT, DG>, dim3(grid),
                         dim3(static_cast<unsigned>(threads)), smem, s, dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part);
    if (e != cudaSuccess || !DG) return e;
    const dim3 rgrid(static_cast<unsigned>(std::max<int64_t>(1, (D + kRedCols - 1) / kRedCols))),
        rblock(kRedCols * kRedSlices);
    return launch_dependent(rmsnorm_dgamma_reduce, rgrid, rblock, 0, s, part, grid, D, dgamma);
}

bool g_fwd_attr[64][4] = {};

template <int ES, int VPT>
cudaError_t launch_fwd_cta_ring(const char* x, int64_t ldx, const char* g, int64_t N, int64_t D, float eps, char* y,
                                int64_t ldy, float* rstd, cudaStream_t s) {
    const int64_t nvec = D / (16 / ES);
    const int threads = static_cast<int>(((nvec + VPT - 1) / VPT + 31) / 32 * 32);
    const size_t smem = static_cast<size_t>(kRingStages) * kRingRows * VPT * threads * 16;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_ring_mu);
        const int k = (ES == 2 ? 0 : 2) + (VPT == kRingVptWide ? 1 : 0);
        if (!g_fwd_attr[dev][k]) {
            e = cudaFuncSetAttribute(rmsnorm_fwd_cta_ring_kernel<ES, kRingRows, VPT>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemMax);
            if (e != cudaSuccess) return e;
            g_fwd_attr[dev][k] = true;
        }
    }
    int per_sm = 0;  // every CTA resident at once: the row ranges are contiguous
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rmsnorm_fwd_cta_ring_kernel<ES, kRingRows, VPT>, threads,
                                                      smem);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(std::min<int64_t>(N, static_cast<int64_t>(device_sm_count()) * std::max(per_sm, 1)));
    return launch_dependent(rmsnorm_fwd_cta_ring_kernel<ES, kRingRows, VPT>, dim3(grid),
                            dim3(static_cast<unsigned>(threads)), smem, s, x, ldx, g, N, D, eps, y, ldy, rstd);
}

}  // namespace

cudaError_t launch_rmsnorm_fwd(int es, const void* X, int64_t ldx, const void* gamma, int64_t N, int64_t D,
                               float eps, void* Y, int64_t ldy, float* rstd, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(norm_grid(N))), block(kNormThreads);
    const char* x = static_cast<const char*>(X);
    const char* g = static_cast<const char*>(gamma);
    char* y = static_cast<char*>(Y);
    // rows of at most 256 vectors (D <= 2048 bf16 / 1024 fp32) in one warp's registers
    const int64_t nvec = D / (16 / es);
    if (nvec <= 128)
        return es == 2 ? launch_dependent(rmsnorm_fwd_reg_kernel<2, 4>, grid, block, 0, s, x, ldx, g, N, D, eps, y, ldy, rstd)
                       : launch_dependent(rmsnorm_fwd_reg_kernel<4, 4>, grid, block, 0, s, x, ldx, g, N, D, eps, y, ldy, rstd);
    if (nvec <= 256)  // (16 vectors a lane held, 8 used: 17.7 us at 8192 x 2048 bf16 against 18.6 with 8)
        return es == 2 ? launch_dependent(rmsnorm_fwd_reg_kernel<2, 16>, grid, block, 0, s, x, ldx, g, N, D, eps, y, ldy, rstd)
                       : launch_dependent(rmsnorm_fwd_reg_kernel<4, 16>, grid, block, 0, s, x, ldx, g, N, D, eps, y, ldy, rstd);
    // up to 1024 vectors (D <= 8192 bf16 / 4096 fp32): the CTA-wide ring
    if (nvec <= static_cast<int64_t>(kRingVpt) * kRingMaxThreads)
        return es == 2 ? launch_fwd_cta_ring<2, kRingVpt>(x, ldx, g, N, D, eps, y, ldy, rstd, s)
                       : launch_fwd_cta_ring<4, kRingVpt>(x, ldx, g, N, D, eps, y, ldy, rstd, s);
    if (nvec <= static_cast<int64_t>(kRingVptWide) * kRingMaxThreads)
        return es == 2 ? launch_fwd_cta_ring<2, kRingVptWide>(x, ldx, g, N, D, eps, y, ldy, rstd, s)
                       : launch_fwd_cta_ring<4, kRingVptWide>(x, ldx, g, N, D, eps, y, ldy, rstd, s);
    return es == 2 ? launch_dependent(rmsnorm_fwd_kernel<2>, grid, block, 0, s, x, ldx, g, N, D, eps, y, ldy, rstd)
                   : launch_dependent(rmsnorm_fwd_kernel<4>, grid, block, 0, s, x, ldx, g, N, D, eps, y, ldy, rstd);
}

cudaError_t launch_rmsnorm_bwd(int es, const void* dY, int64_t lddy, const void* X, int64_t ldx, const void* gamma,
                               const float* rstd, int64_t N, int64_t D, void* dX, int64_t lddx, float* part,
                               float* dgamma, cudaStream_t s) {
    const int64_t nvec = D / (16 / es);
    const char* dy = static_cast<const char*>(dY);
    const char* x = static_cast<const char*>(X);
    const char* g = static_cast<const char*>(gamma);
    char* dx = static_cast<char*>(dX);
    const dim3 rgrid(static_cast<unsigned>(std::max<int64_t>(1, (D + kRedCols - 1) / kRedCols))),
        rblock(kRedCols * kRedSlices);
    cudaError_t e = cudaSuccess;
    if (N > 0 && nvec <= static_cast<int64_t>(kRingVptWide) * kRingMaxThreads) {
        const bool narrow = nvec <= static_cast<int64_t>(kRingVpt) * kRingMaxThreads;
        if (es == 2) {
            if (narrow)
                return dgamma ? launch_bwd_ring<2, kRingVpt, true>(dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part, dgamma, s)
                              : launch_bwd_ring<2, kRingVpt, false>(dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part, dgamma, s);
            return dgamma ? launch_bwd_ring<2, kRingVptWide, true>(dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part, dgamma, s)
                          : launch_bwd_ring<2, kRingVptWide, false>(dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part, dgamma, s);
        }
        if (narrow)
            return dgamma ? launch_bwd_ring<4, kRingVpt, true>(dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part, dgamma, s)
                          : launch_bwd_ring<4, kRingVpt, false>(dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part, dgamma, s);
        return dgamma ? launch_bwd_ring<4, kRingVptWide, true>(dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part, dgamma, s)
                      : launch_bwd_ring<4, kRingVptWide, false>(dy, lddy, x, ldx, g, rstd, N, D, dx, lddx, part, dgamma, s);
    }
    if (N > 0) {
        const dim3 grid(static_cast<unsigned>(norm_grid(N))), block(kNormThreads);
        e = es == 2 ? launch_dependent(rmsnorm_bwd_kernel<2>, grid, block, 0, s, dy, lddy, x, ldx, g, rstd, N, D, dx, lddx)
                    : launch_dependent(rmsnorm_bwd_kernel<4>, grid, block, 0, s, dy, lddy, x, ldx, g, rstd, N, D, dx, lddx);
        if (e != cudaSuccess) return e;
    }
    if (!dgamma) return cudaSuccess;
    const int epv = 16 / es;
    const dim3 ggrid(static_cast<unsigned>((D / epv + kGammaThreads - 1) / kGammaThreads), kRmsGammaGroups);
    e = es == 2 ? launch_dependent(rmsnorm_dgamma_kernel<2>, ggrid, dim3(kGammaThreads), 0, s, dy, lddy, x, ldx, rstd, N,
                                   D, part)
                : launch_dependent(rmsnorm_dgamma_kernel<4>, ggrid, dim3(kGammaThreads), 0, s, dy, lddy, x, ldx, rstd, N,
                                   D, part);
    if (e != cudaSuccess) return e;
    return launch_dependent(rmsnorm_dgamma_reduce, rgrid, rblock, 0, s, part, static_cast<int>(kRmsGammaGroups), D,
                            dgamma);
}

}  // namespace foak
