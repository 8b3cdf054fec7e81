// Cross-entropy backward from a saved log-sum-exp:
//   dlogits_ij = (exp(x_ij - lse_i) - [j == y_i]) * g / D,  ignored rows +0.0.
// With lse known every element is independent, so this is a pure stream over
// (row, 32 KB segment) work items: each thread issues its 8 x 16-byte loads
// first, then computes and stores.  Ignored rows are never read.  This is the
// separate backward of the FastCrossEntropyLoss pair (fms-acceleration PR #79,
// Description item 4); the fused kernel in ce_rows.cu avoids its second read.
#include <algorithm>

#include "common.cuh"
#include "foak_ce.h"
#include "internal.h"

namespace foak {

constexpr int kBwdThreads = 256;
constexpr int kBwdVpt = 8;
constexpr int kBwdSegVec = kBwdThreads * kBwdVpt;  // 2048 vectors = 32 KB
constexpr int kBwdBlocksPerSm = 4;

struct CeBwdParams {
    const char* x;
    char* dx;
    int64_t ld;
    const int64_t* labels;
    int64_t N, V, ignore_index;
    const float* lse;
    const float* g_ptr;    // device g; null: g_host
    float g_host;
    float denom;
    const int64_t* denom_dev;  // if set: the denominator, read from device memory
    int32_t* err;
    int64_t nseg;
};

template <int ES>
__device__ __forceinline__ float bwd_load_scalar(const char* p) {
    if constexpr (ES == 2) return bf16_lo(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)));
    else return *reinterpret_cast<const float*>(p);
}

template <int ES>
__device__ __forceinline__ void bwd_store_scalar(char* p, float v) {
    if constexpr (ES == 2) *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
    else *reinterpret_cast<float*>(p) = v;
}

template <int ES>
__global__ void __launch_bounds__(kBwdThreads) ce_backward_kernel(const CeBwdParams p) {
    griddep_launch_dependents();  // programmatic dependent launch: no global access before the wait
    griddep_wait();
    constexpr int EPV = 16 / ES;
    __shared__ int iscratch[2 * (kBwdThreads / 32)];
    const int tid = threadIdx.x;

    int n_valid = 0, n_bad = 0;
    if ((!p.denom_dev && p.denom <= 0.f) || blockIdx.x == 0)
        count_labels(p.labels, p.N, p.V, p.ignore_index, iscratch, n_valid, n_bad);
    if (blockIdx.x == 0 && tid == 0 && p.err) *p.err = n_bad > 0 ? FOAK_ERRBIT_LABEL_RANGE : 0;
    const float g = p.g_ptr ? __ldg(p.g_ptr) : p.g_host;
    const float D = p.denom_dev ? static_cast<float>(__ldg(p.denom_dev))
                                : (p.denom > 0.f ? p.denom : static_cast<float>(n_valid));
    const float scale = g / D;
    const int64_t row_bytes = p.ld * ES;
    const int64_t items = p.N * p.nseg;

    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t row = item / p.nseg;
        const int64_t seg = item - row * p.nseg;
        const int64_t y = __ldg(p.labels + row);
        const bool valid = y != p.ignore_index && y >= 0 && y < p.V;
        const char* rowp = p.x + row * row_bytes;
        char* drow = p.dx + row * row_bytes;
        int h = static_cast<int>(((16u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(rowp)) & 15u)) & 15u) / ES);
        if (h > p.V) h = static_cast<int>(p.V);
        const int64_t nb = (p.V - h) / EPV;
        const int t = static_cast<int>(p.V - h - nb * EPV);
        const int64_t tail_col = h + nb * EPV;
        const int64_t vbeg = seg * kBwdSegVec;
        const int64_t vend = std::min<int64_t>(nb, vbeg + kBwdSegVec);
        const uint4* src = reinterpret_cast<const uint4*>(rowp + static_cast<int64_t>(h) * ES);
        uint4* dst = reinterpret_cast<uint4*>(drow + static_cast<int64_t>(h) * ES);
        // scalar head (segment 0, thread 0) and tail (last segment, thread 1)
        const bool do_head = seg == 0 && tid == 0 && h > 0;
        const bool do_tail = seg == p.nseg - 1 && tid == 1 && t > 0;

        if (!valid) {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int64_t vv = vbeg + tid; vv < vend; vv += kBwdThreads) st_global_cs_v4(dst + vv, z);
            if (do_head)
                for (int s = 0; s < h; ++s) bwd_store_scalar<ES>(drow + s * ES, 0.f);
            if (do_tail)
                for (int s = 0; s < t; ++s) bwd_store_scalar<ES>(drow + (tail_col + s) * ES, 0.f);
            continue;
        }
        const float c = __ldg(p.lse + row) * kLog2e;
        int64_t yvec = -1;
        int ye = 0;
        if (y >= h && y < tail_col) {
            yvec = (y - h) / EPV;
            ye = static_cast<int>((y - h) % EPV);
        }
        uint4 v[kBwdVpt];
#pragma unroll
        for (int i = 0; i < kBwdVpt; ++i) {
            const int64_t vv = vbeg + tid + i * kBwdThreads;
            if (vv < vend) v[i] = ld_global_v4(src + vv);
        }
#pragma unroll
        for (int i = 0; i < kBwdVpt; ++i) {
            const int64_t vv = vbeg + tid + i * kBwdThreads;
            if (vv < vend) {
                float f[EPV], d[EPV];
                if constexpr (ES == 2) {
                    f[0] = bf16_lo(v[i].x); f[1] = bf16_hi(v[i].x);
                    f[2] = bf16_lo(v[i].y); f[3] = bf16_hi(v[i].y);
                    f[4] = bf16_lo(v[i].z); f[5] = bf16_hi(v[i].z);
                    f[6] = bf16_lo(v[i].w); f[7] = bf16_hi(v[i].w);
                } else {
                    f[0] = __uint_as_float(v[i].x); f[1] = __uint_as_float(v[i].y);
                    f[2] = __uint_as_float(v[i].z); f[3] = __uint_as_float(v[i].w);
                }
#pragma unroll
                for (int e = 0; e < EPV; ++e) d[e] = ex2(fmaf(f[e], kLog2e, -c)) * scale;
                if (vv == yvec) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (e == ye) d[e] -= scale;
                }
                uint4 o;
                if constexpr (ES == 2) {
                    o.x = pack_bf16x2(d[0], d[1]);
                    o.y = pack_bf16x2(d[2], d[3]);
                    o.z = pack_bf16x2(d[4], d[5]);
                    o.w = pack_bf16x2(d[6], d[7]);
                } else {
                    o.x = __float_as_uint(d[0]); o.y = __float_as_uint(d[1]);
                    o.z = __float_as_uint(d[2]); o.w = __float_as_uint(d[3]);
                }
                st_global_cs_v4(dst + vv, o);
            }
        }
        if (do_head) {
            for (int s = 0; s < h; ++s) {
                float d = ex2(fmaf(bwd_load_scalar<ES>(rowp + s * ES), kLog2e, -c)) * scale;
                if (s == y) d -= scale;
                bwd_store_scalar<ES>(drow + s * ES, d);
            }
        }
        if (do_tail) {
            for (int s = 0; s < t; ++s) {
                const int64_t col = tail_col + s;
                float d = ex2(fmaf(bwd_load_scalar<ES>(rowp + col * ES), kLog2e, -c)) * scale;
                if (col == y) d -= scale;
                bwd_store_scalar<ES>(drow + col * ES, d);
            }
        }
    }
}

cudaError_t launch_ce_backward(int elem_bytes, void* dx, const void* x, int64_t ld,
                               const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index,
                               const float* lse, const float* g_ptr, float denom, int32_t* err,
                               cudaStream_t stream, float g_host, const int64_t* denom_dev) {
    CeBwdParams prm = {};
    prm.x = static_cast<const char*>(x);
    prm.dx = static_cast<char*>(dx);
    prm.ld = ld;
    prm.labels = labels;
    prm.N = N;
    prm.V = V;
    prm.ignore_index = ignore_index;
    prm.lse = lse;
    prm.g_ptr = g_ptr;
    prm.g_host = g_host;
    prm.denom = denom;
    prm.denom_dev = denom_dev;
    prm.err = err;
    const int64_t nb_max = V * elem_bytes / 16;
    prm.nseg = std::max<int64_t>(1, (nb_max + kBwdSegVec - 1) / kBwdSegVec);
    const int64_t items = N * prm.nseg;
    const int64_t full = static_cast<int64_t>(device_sm_count()) * kBwdBlocksPerSm;
    const unsigned grid = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(full, items)));
    return elem_bytes == 2 ? launch_dependent(ce_backward_kernel<2>, dim3(grid), dim3(kBwdThreads), 0, stream, prm)
                           : launch_dependent(ce_backward_kernel<4>, dim3(grid), dim3(kBwdThreads), 0, stream, prm);
}

}  // namespace foak
