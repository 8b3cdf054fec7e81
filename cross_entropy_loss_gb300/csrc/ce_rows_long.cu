// Row-wise cross-entropy for rows longer than one CTA's 64 KB slice, without
// clusters: one 512-thread CTA owns a whole row and streams it through a ring
// of 64 KB shared-memory stages (one-dimensional bulk copies completing on
// mbarriers) twice.
//
//   pass 1  every thread folds its share of each chunk into a running
//           (max, sum exp(x - max)) -- the max is kept per warp, so a chunk
//           costs one warp shuffle-max and one rescale -- and the CTA merges
//           the pairs once, at the row's end, into the log-sum-exp;
//   pass 2  (fused forward+backward) the same chunks are loaded again and
//           (exp(x - lse) - onehot) * g / D is written over them with 16-byte
//           streaming stores.
//
// A row is 250 KB (bf16) or 501 KB (fp32) at V = 128256; 152 CTAs hold about
// 40 or 80 MB of rows between the two passes, well inside the 129 MB L2, so the
// second read is served from L2 and HBM sees each logit read once and written
// once, as in the one-pass kernel.  Against a cluster per row this uses every
// SM (clusters of 4 or 8 do not tile 152 SMs), needs no distributed shared
// memory exchange, and pays the CTA-wide reduction once per row instead of
// once per 64 KB slice.  It is the same two-sweep row computation as the
// FastCrossEntropyLoss kernel of the FOAK pages (fms-acceleration PR #79,
// Description item 4: log-sum-exp first, then the gradient in place), with
// the row split into chunks where the original holds it in one block.
#include <algorithm>
#include <mutex>
#include <map>

#include "row_common.cuh"

namespace foak {

namespace {

constexpr int kLongThreads = 512;
constexpr int kLongWarps = kLongThreads / 32;
constexpr int kLongVpt = 8;
constexpr int kLongChunkVec = kLongThreads * kLongVpt;  // 4096 vectors = 64 KB
constexpr int kLongChunkShift = 12;
static_assert(kLongChunkVec == 1 << kLongChunkShift, "chunk is a power of two");

__device__ __forceinline__ bool label_valid(int64_t y, const CeRowParams& p) {
    return y != p.ignore_index && y >= 0 && y < p.V;
}

template <int ES, bool GRAD>
__global__ void __launch_bounds__(kLongThreads, 1) ce_rows_long_kernel(const CeRowParams p) {
    constexpr int THREADS = kLongThreads, VPT = kLongVpt, WARPS = kLongWarps, EPV = 16 / ES;
    constexpr int PASSES = GRAD ? 2 : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bars[kRowMaxStages];
    __shared__ float2 red_ms[2][WARPS];
    __shared__ int64_t s_lab[kLabCache];
    __shared__ int iscratch[2 * WARPS];
    __shared__ double dred[WARPS];
    __shared__ int s_abort, s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t cid = blockIdx.x, ncl = gridDim.x;
    const int64_t n_it = p.N > cid ? (p.N - 1 - cid) / ncl + 1 : 0;
    const int64_t row_bytes = p.ld * ES;
    const int S = p.stages;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        s_abort = 0;
        s_last = 0;
    }
    __syncthreads();

    bool lab_cached = false;
    auto label_of = [&](int64_t it) -> int64_t {
        return (lab_cached && it < kLabCache) ? s_lab[it] : __ldg(p.labels + cid + it * ncl);
    };

    // Producer (thread 0).  The load sequence is: for every valid row, its
    // chunks for pass 1, then (fused) the same chunks again for pass 2.
    int64_t p_it = -1;      // row iteration being loaded
    int p_pass = 0, p_chunk = 0, p_nchunk = 0;
    const char* p_src = nullptr;
    int64_t p_nb = 0;
    uint32_t p_v = 0;       // chunk loads issued (one stage each)
    auto issue_next = [&]() {
        while (true) {
            const bool row_done = p_it < 0 || p_nchunk == 0 || (p_pass == PASSES - 1 && p_chunk == p_nchunk - 1);
            if (row_done) {
                int64_t it = p_it + 1;
                while (it < n_it && !label_valid(label_of(it), p)) ++it;
                p_it = it;
                p_nchunk = 0;
                if (it >= n_it) return;
                const char* rowp = p.x + (cid + it * ncl) * row_bytes;
                const RowGeom gm = row_geom<ES>(rowp, p.V);
                p_src = rowp + static_cast<int64_t>(gm.h) * ES;
                p_nb = gm.nb;
                p_nchunk = static_cast<int>((gm.nb + kLongChunkVec - 1) >> kLongChunkShift);
                p_pass = 0;
                p_chunk = 0;
                if (p_nchunk == 0) continue;  // scalars only: nothing to stream
                if (p.skip_load_row == cid + it * ncl) {  // test hook: this stage never completes
                    ++p_v;
                    return;
                }
            } else if (p_chunk == p_nchunk - 1) {
                ++p_pass;
                p_chunk = 0;
            } else {
                ++p_chunk;
            }
            const int64_t c0 = static_cast<int64_t>(p_chunk) << kLongChunkShift;
            const int64_t nl = std::min<int64_t>(kLongChunkVec, p_nb - c0);
            const uint32_t bytes = static_cast<uint32_t>(nl) * 16u;
            const int st = static_cast<int>(p_v % static_cast<uint32_t>(S));
            ++p_v;
            mbar_arrive_expect_tx(&bars[st], bytes);
            unsigned char* dst = smem + static_cast<size_t>(st) * p.stage_bytes;
            for (uint32_t off = 0; off < bytes; off += kBulkChunk)
                bulk_g2s(dst + off, p_src + c0 * 16 + off, min(kBulkChunk, bytes - off), &bars[st]);
            return;
        }
    };
    if (tid == 0)
        for (int s = 0; s < S; ++s) issue_next();

    int n_valid = 0, n_bad = 0;
    count_labels(p.count_labels, p.count_N, p.V, p.ignore_index, iscratch, n_valid, n_bad);
    const float D = p.denom > 0.f ? p.denom : static_cast<float>(n_valid);
    const float scale = p.g / D;
    for (int64_t it = tid; it < n_it && it < kLabCache; it += THREADS) s_lab[it] = __ldg(p.labels + cid + it * ncl);
    __syncthreads();
    lab_cached = true;

    // For scale > 0 the scale is folded into the exponent; otherwise multiplied.
    const bool mul = !(scale > 0.f);
    const float log2_scale = mul ? 0.f : log2f(scale);

    uint32_t c_v = 0;   // chunks consumed
    uint32_t c_ok = 0;  // chunks whose load was seen complete (a prefix of the loads)
    uint32_t n_rows = 0;
    bool aborted = false;
    const uint4 pad = RowMath<ES>::pad();

    // Wait for the next chunk and move it into registers (-inf past its end).
    auto take_chunk = [&](int nl, uint4 (&v)[VPT]) {
        const int st = static_cast<int>(c_v % static_cast<uint32_t>(S));
        const uint32_t par = (c_v / static_cast<uint32_t>(S)) & 1u;
        ++c_v;
        if (!aborted) {
            if (mbar_wait_bounded(&bars[st], par, p.wait_ns)) c_ok = c_v;
            else s_abort = 1;
        }
        const uint4* sb = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(st) * p.stage_bytes);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int lv = tid + i * THREADS;
            v[i] = lv < nl ? sb[lv] : pad;
        }
    };
    // After every thread has its copy: pick up an abort, refill the freed stage.
    auto release = [&]() {
        if (s_abort) aborted = true;
        if (tid == 0 && !aborted) {
            fence_proxy_async_smem();
            issue_next();
        }
    };

    for (int64_t it = 0; it < n_it; ++it) {
        const int64_t row = cid + it * ncl;
        const int64_t y = label_of(it);
        const char* rowp = p.x + row * row_bytes;
        const RowGeom gm = row_geom<ES>(rowp, p.V);
        const int nchunk = static_cast<int>((gm.nb + kLongChunkVec - 1) >> kLongChunkShift);
        const bool has_head = tid == 0 && gm.h > 0;
        const bool has_tail = tid == 32 && gm.t > 0;  // another warp than the head's
        const int64_t tail_col = gm.h + gm.nb * EPV;
        const int ns = has_head ? gm.h : (has_tail ? gm.t : 0);
        const int64_t sc0 = has_head ? 0 : tail_col;

        if (!label_valid(y, p)) {
            if constexpr (GRAD) {
                char* drow = p.dx + row * row_bytes;
                uint4* dv = reinterpret_cast<uint4*>(drow + static_cast<int64_t>(gm.h) * ES);
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                for (int64_t i = tid; i < gm.nb; i += THREADS) st_global_cs_v4(dv + i, z);
                for (int s = 0; s < ns; ++s) store_scalar<ES>(drow + (sc0 + s) * ES, 0.f);
            }
            if (tid == 0) {
                p.row_loss[row] = 0.f;
                if (p.lse) p.lse[row] = 0.f;
            }
            continue;
        }
        const int rb = n_rows & 1u;  // red_ms is double-buffered by row parity
        ++n_rows;

        // Where the label column lives: a scalar of the head or tail, or element
        // own_e of vector own_slot of chunk own_chunk in this thread's registers.
        int own_chunk = -1, own_slot = -1, own_e = 0, own_sc = -1;
        if (y < gm.h) {
            if (tid == 0) own_sc = static_cast<int>(y);
        } else if (y < tail_col) {
            const int64_t ly = y - gm.h;
            const int64_t lvec = ly / EPV;
            const int lv = static_cast<int>(lvec & (kLongChunkVec - 1));
            if ((lv & (THREADS - 1)) == tid) {
                own_chunk = static_cast<int>(lvec >> kLongChunkShift);
                own_slot = lv / THREADS;
                own_e = static_cast<int>(ly % EPV);
            }
        } else if (tid == 32) {
            own_sc = static_cast<int>(y - tail_col);
        }

        // ---- pass 1: running (max, sum) per thread, max shared by the warp
        float M = kNegInf, s = 0.f, x_y = 0.f;
        float xs[kMaxScalars];
        if (gm.h > 0 || gm.t > 0) {  // CTA-uniform
            float xm = kNegInf;
            if (ns > 0) {
#pragma unroll
                for (int q = 0; q < kMaxScalars; ++q) {
                    xs[q] = q < ns ? load_scalar<ES>(rowp + (sc0 + q) * ES) : kNegInf;
                    xm = fmaxf(xm, xs[q]);
                }
            }
            M = warp_max(xm);
            if (ns > 0) {
                const float mb = M == kNegInf ? 0.f : M * kLog2e;
#pragma unroll
                for (int q = 0; q < kMaxScalars; ++q) {
                    if (q < ns) s += ex2(fmaf(xs[q], kLog2e, -mb));
                    if (q == own_sc) x_y = xs[q];
                }
            }
        }
        for (int j = 0; j < nchunk; ++j) {
            const int nl = static_cast<int>(std::min<int64_t>(kLongChunkVec, gm.nb - (static_cast<int64_t>(j) << kLongChunkShift)));
            uint4 v[VPT];
            take_chunk(nl, v);
            const bool last = j == nchunk - 1;
            if (!last) {
                __syncthreads();
                release();
            }
            const float Mn = fmaxf(M, warp_max(RowMath<ES>::template vmax<VPT>(v)));
            if (Mn != M) s *= ex2((M - Mn) * kLog2e);
            M = Mn;
            s += RowMath<ES>::template vsum<VPT>(v, M == kNegInf ? 0.f : M * kLog2e);
            if (j == own_chunk) {
#pragma unroll
                for (int i = 0; i < VPT; ++i)
                    if (i == own_slot) x_y = vec_elem<ES>(v[i], own_e);
            }
            if (last) {
                const float sw = warp_sum(s);
                if (lane == 0) red_ms[rb][warp] = make_float2(M, sw);
                __syncthreads();
                release();
            }
        }
        if (nchunk == 0) {
            const float sw = warp_sum(s);
            if (lane == 0) red_ms[rb][warp] = make_float2(M, sw);
            __syncthreads();
            if (s_abort) aborted = true;
        }
        const float2 pr = lane < WARPS ? red_ms[rb][lane] : make_float2(kNegInf, 0.f);
        const float Mr = warp_max(pr.x);
        const float Sr = warp_sum(pr.x == kNegInf ? 0.f : pr.y * ex2((pr.x - Mr) * kLog2e));
        const float lse2 = fmaf(Mr, kLog2e, lg2(Sr));  // log-sum-exp in base 2
        const float lse = lse2 * kLn2;
        if ((own_chunk >= 0 || own_sc >= 0) && !aborted) p.row_loss[row] = lse - x_y;
        if (tid == 0 && p.lse && !aborted) p.lse[row] = lse;

        // ---- pass 2: gradient over the same chunks, reloaded
        if constexpr (GRAD) {
            const float c = lse2 - log2_scale;
            const f32x2_t L2 = f2_pack(kLog2e, kLog2e), C2 = f2_pack(-c, -c), S2 = f2_pack(scale, scale);
            char* drow = p.dx + row * row_bytes;
            uint4* dv = reinterpret_cast<uint4*>(drow + static_cast<int64_t>(gm.h) * ES);
            for (int j = 0; j < nchunk; ++j) {
                const int64_t cv0 = static_cast<int64_t>(j) << kLongChunkShift;
                const int nl = static_cast<int>(std::min<int64_t>(kLongChunkVec, gm.nb - cv0));
                uint4 v[VPT];
                take_chunk(nl, v);
                __syncthreads();
                release();
                if (aborted) continue;
                const int slot = j == own_chunk ? own_slot : -1;
                uint4* dvc = dv + cv0;
                if (!mul) {
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        const int lv = tid + i * THREADS;
                        uint4 o = RowMath<ES>::template vexp<false>(v[i], L2, C2, S2);
                        if (i == slot) o = vec_grad_label<ES>(v[i], own_e, c, false, scale);
                        if (lv < nl) st_global_cs_v4(dvc + lv, o);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        const int lv = tid + i * THREADS;
                        uint4 o = RowMath<ES>::template vexp<true>(v[i], L2, C2, S2);
                        if (i == slot) o = vec_grad_label<ES>(v[i], own_e, c, true, scale);
                        if (lv < nl) st_global_cs_v4(dvc + lv, o);
                    }
                }
            }
            if (ns > 0 && !aborted) {
#pragma unroll
                for (int q = 0; q < kMaxScalars; ++q) {
                    if (q < ns) {
                        float d = ex2(fmaf(xs[q], kLog2e, -c));
                        if (mul) d *= scale;
                        if (q == own_sc) d -= scale;
                        store_scalar<ES>(drow + (sc0 + q) * ES, d);
                    }
                }
            }
        }
    }

    // After an abort, loads issued past the last one seen complete may still be
    // landing in shared memory: wait for them (bounded) before the CTA exits.
    if (tid == 0) {
        for (uint32_t k = c_ok; k < p_v; ++k)
            (void)mbar_wait_bounded(&bars[k % static_cast<uint32_t>(S)], (k / static_cast<uint32_t>(S)) & 1u,
                                    p.wait_ns);
    }
    rows_finish<THREADS>(p, aborted, n_valid, n_bad, &s_last, dred);
}

std::mutex g_long_mu;
std::map<std::pair<int, const void*>, bool> g_long_attr;  // (device, kernel): smem limit raised

template <int ES, bool GRAD>
cudaError_t launch_long_typed(const CeRowParams& base, cudaStream_t stream) {
    const void* kern = reinterpret_cast<const void*>(&ce_rows_long_kernel<ES, GRAD>);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(g_long_mu);
        bool& set = g_long_attr[std::make_pair(dev, kern)];
        if (!set) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBudget));
            if (e != cudaSuccess) return e;
            set = true;
        }
    }
    CeRowParams prm = base;
    prm.k = 1;
    prm.per = kLongChunkVec;
    prm.stage_bytes = kLongChunkVec * 16;
    prm.stages = static_cast<int>(std::min<size_t>(kRowMaxStages, kSmemBudget / prm.stage_bytes));
    const size_t smem = static_cast<size_t>(prm.stages) * prm.stage_bytes;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(device_sm_count(), base.N));
    ce_rows_long_kernel<ES, GRAD><<<static_cast<unsigned>(grid), kLongThreads, smem, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ce_rows_long(bool grad, int elem_bytes, const CeRowParams& base, cudaStream_t stream) {
    if (elem_bytes == 2) return grad ? launch_long_typed<2, true>(base, stream) : launch_long_typed<2, false>(base, stream);
    return grad ? launch_long_typed<4, true>(base, stream) : launch_long_typed<4, false>(base, stream);
}

}  // namespace foak
