// Rotary position embedding -- the "Fast RoPE" kernel the FOAK pages list among
// their fused operations (fms-acceleration-foak 0.7.4 page), here with the explicit
// position ids the pages note the FOAK version lacks (foak page, Known Issues;
// fms-hf-tuning PR #280, Notes on FastKernels).  The pages print no formula; the
// operation is the Llama / Mistral rotary embedding in the "rotate half" pairing:
// for head dimension d and i < d/2, elements i and i + d/2 of every head vector of
// token t turn by theta = p_t * base^(-2i/d):
//     x'_i = x_i cos(theta) - x_{i+d/2} sin(theta),  x'_{i+d/2} = x_{i+d/2} cos(theta) + x_i sin(theta)
// and the backward turns by -theta (the rotation's transpose).
//
// The angles are not formed in fp32 on the fly: at position 8192 an fp32 theta is
// off by up to 5e-4 rad.  rope_cache_kernel builds cos and sin for every (position,
// frequency) once, in float64 (the angle and its reduction), stored as fp32; the
// apply kernel gathers its token's row of the table (L2-resident: 4 MB for 8192
// positions at d = 128).  The apply kernel is HBM-bound: each element read and
// written once, in place.  One thread owns a pair of 16-byte vectors -- elements
// i..i+EPV-1 and the same run shifted by d/2 -- of one head of one token.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "foak_ce.h"
#include "internal.h"

namespace foak {

namespace {

constexpr int kRopeThreads = 256;

// cos_t[p * half + i], sin_t[p * half + i] for p < P, i < half = d / 2.
__global__ void rope_cache_kernel(double log2_base, int d, int64_t P, float* __restrict__ cos_t,
                                  float* __restrict__ sin_t) {
    const int half = d / 2;
    const int64_t n = P * half;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t p = idx / half;
        const int i = static_cast<int>(idx - p * half);
        const double inv_freq = exp2(-2.0 * static_cast<double>(i) / static_cast<double>(d) * log2_base);
        const double theta = static_cast<double>(p) * inv_freq;
        double s, c;
        sincos(theta, &s, &c);
        cos_t[idx] = static_cast<float>(c);
        sin_t[idx] = static_cast<float>(s);
    }
}

template <int ES>
__device__ __forceinline__ void ld8(const char* p, float (&f)[16 / ES]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    if constexpr (ES == 2) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
}

template <int ES>
__device__ __forceinline__ void st8(char* p, const float (&f)[16 / ES]) {
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

// Up to two tensors (Q and K) in one launch: tensor k is T tokens x H[k] heads x d,
// token stride ldt[k] elements, heads contiguous (stride d).
struct RopeTensors {
    char* X[2];
    int H[2];
    int64_t ldt[2];
};

template <int ES>
__global__ void __launch_bounds__(kRopeThreads) rope_apply_kernel(const RopeTensors a, int64_t T, int d,
                                                                  const int64_t* __restrict__ positions,
                                                                  const float* __restrict__ cos_t,
                                                                  const float* __restrict__ sin_t, int64_t P,
                                                                  float sign, int32_t* err) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    constexpr int EPV = 16 / ES;
    const int half = d / 2;
    const int per_head = half / EPV;  // vector pairs per head
    const int64_t n0 = T * a.H[0] * per_head;
    const int64_t n = n0 + T * a.H[1] * per_head;
    for (int64_t w0 = blockIdx.x * static_cast<int64_t>(kRopeThreads) + threadIdx.x; w0 < n;
         w0 += static_cast<int64_t>(gridDim.x) * kRopeThreads) {
        const int which = w0 < n0 ? 0 : 1;
        const int64_t w = which ? w0 - n0 : w0;
        const int H = a.H[which];
        const int64_t ldt = a.ldt[which];
        char* X = a.X[which];
        const int j = static_cast<int>(w % per_head);
        const int64_t th = w / per_head;
        const int h = static_cast<int>(th % H);
        const int64_t t = th / H;
        // the data loads do not depend on the position: they go out with its load
        char* lo_p = X + ((t * ldt) + static_cast<int64_t>(h) * d + static_cast<int64_t>(j) * EPV) * ES;
        char* hi_p = lo_p + static_cast<int64_t>(half) * ES;
        float lo[EPV], hi[EPV], c[EPV], s[EPV];
        const int64_t p = __ldg(positions + t);
        ld8<ES>(lo_p, lo);
        ld8<ES>(hi_p, hi);
        if (p < 0 || p >= P) {  // left untouched, flagged
            if (err && j == 0 && h == 0) atomicOr(reinterpret_cast<unsigned*>(err), FOAK_ERRBIT_LABEL_RANGE);
            continue;
        }
        const float* cr = cos_t + p * half + j * EPV;
        const float* sr = sin_t + p * half + j * EPV;
#pragma unroll
        for (int k = 0; k < EPV; k += 4) {
            const float4 c4 = __ldg(reinterpret_cast<const float4*>(cr + k));
            const float4 s4 = __ldg(reinterpret_cast<const float4*>(sr + k));
            c[k] = c4.x; c[k + 1] = c4.y; c[k + 2] = c4.z; c[k + 3] = c4.w;
            s[k] = sign * s4.x; s[k + 1] = sign * s4.y; s[k + 2] = sign * s4.z; s[k + 3] = sign * s4.w;
        }
        float olo[EPV], ohi[EPV];
#pragma unroll
        for (int k = 0; k < EPV; ++k) {
            olo[k] = fmaf(lo[k], c[k], -hi[k] * s[k]);
            ohi[k] = fmaf(hi[k], c[k], lo[k] * s[k]);
        }
        st8<ES>(lo_p, olo);
        st8<ES>(hi_p, ohi);
    }
}

}  // namespace

size_t rope_cache_bytes(int64_t max_pos, int d) {
    return 2 * ((static_cast<size_t>(max_pos) * static_cast<size_t>(d / 2) * 4 + 255) / 256 * 256);
}

cudaError_t launch_rope_cache(double base, int d, int64_t max_pos, void* cache, cudaStream_t s) {
    if (max_pos == 0) return cudaSuccess;
    float* cos_t = static_cast<float*>(cache);
    float* sin_t = reinterpret_cast<float*>(static_cast<char*>(cache) + rope_cache_bytes(max_pos, d) / 2);
    const int64_t n = max_pos * (d / 2);
    const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(device_sm_count()) * 16));
    rope_cache_kernel<<<std::max(grid, 1), 256, 0, s>>>(std::log2(base), d, max_pos, cos_t, sin_t);
    return cudaGetLastError();
}

cudaError_t launch_rope_apply(int es, void* X, int64_t T, int H, int64_t ldt, void* X2, int H2, int64_t ldt2, int d,
                              const int64_t* positions, const void* cache, int64_t max_pos, bool inverse,
                              int32_t* err, cudaStream_t s) {
    if (T == 0 || H + H2 == 0) return cudaSuccess;
    const float* cos_t = static_cast<const float*>(cache);
    const float* sin_t =
        reinterpret_cast<const float*>(static_cast<const char*>(cache) + rope_cache_bytes(max_pos, d) / 2);
    RopeTensors a;
    a.X[0] = static_cast<char*>(X);
    a.H[0] = H;
    a.ldt[0] = ldt;
    a.X[1] = static_cast<char*>(X2);
    a.H[1] = X2 ? H2 : 0;
    a.ldt[1] = ldt2;
    const int64_t n = T * (a.H[0] + a.H[1]) * (d / 2 / (16 / es));
    const int grid =
        static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n + kRopeThreads - 1) / kRopeThreads,
                                                                static_cast<int64_t>(device_sm_count()) * 8)));
    const float sign = inverse ? -1.f : 1.f;
    return es == 2 ? launch_dependent(rope_apply_kernel<2>, dim3(grid), dim3(kRopeThreads), 0, s, a, T, d, positions,
                                      cos_t, sin_t, max_pos, sign, err)
                   : launch_dependent(rope_apply_kernel<4>, dim3(grid), dim3(kRopeThreads), 0, s, a, T, d, positions,
                                      cos_t, sin_t, max_pos, sign, err);
}

}  // namespace foak
