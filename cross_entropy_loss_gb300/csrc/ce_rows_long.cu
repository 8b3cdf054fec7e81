// Row-wise cross-entropy for rows longer than one CTA's 64 KB slice, without
// clusters: one CTA owns a whole row and streams it through a ring of
// shared-memory stages (one-dimensional bulk copies completing on mbarriers)
// twice.
//
//   pass 1  every thread folds its share of each chunk into a running
//           (max, sum exp(x - max)) -- the max is kept per warp, so a chunk
//           costs one warp shuffle-max and one rescale -- and the CTA merges
//           the pairs once, at the row's end, into the log-sum-exp;
//   pass 2  (fused forward+backward) the same chunks are loaded again and
//           (exp(x - lse) - onehot) * g / D is written over them with 16-byte
//           streaming stores.
//
// Stages are handed back per warp: the last warp to take a chunk into its
// registers refills the stage, so warps only meet at the one CTA barrier per
// row that merges the (max, sum) pairs.
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
#include <cstdlib>
#include <map>
#include <mutex>

#include "row_common.cuh"

namespace foak {

namespace {

constexpr int kLongMaxStages = 4;

__device__ __forceinline__ bool label_valid(int64_t y, const CeRowParams& p) {
    return y != p.ignore_index && y >= 0 && y < p.V;
}

// THREADS threads x VPT 16-byte vectors per thread = one chunk (48 or 64 KB).
template <int ES, bool GRAD, int THREADS, int VPT>
__global__ void __launch_bounds__(THREADS, 1) ce_rows_long_kernel(const CeRowParams p) {
    constexpr int WARPS = THREADS / 32, EPV = 16 / ES;
    constexpr int CHUNK = THREADS * VPT;  // vectors per chunk
    constexpr int PASSES = GRAD ? 2 : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kLongMaxStages];   // chunk landed (producer's expect_tx + bytes)
    __shared__ unsigned s_rel[kLongMaxStages];  // warps that released each stage, cumulative
    __shared__ unsigned s_iss[kLongMaxStages];  // loads issued into each stage
    __shared__ float2 red_ms[2][WARPS];
    __shared__ int64_t s_lab[kLabCache];
    __shared__ int iscratch[2 * WARPS];
    __shared__ DFloat dred[WARPS];
    __shared__ int s_abort, s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t cid = blockIdx.x, ncl = gridDim.x;
    const int64_t n_it = p.N > cid ? (p.N - 1 - cid) / ncl + 1 : 0;
    const int64_t row_bytes = p.ld * ES;
    const uint32_t S = static_cast<uint32_t>(p.stages);

    if (tid == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            s_rel[s] = 0;
            s_iss[s] = 0;
        }
        fence_mbar_init();
        s_abort = 0;
        s_last = 0;
    }
    // shared memory only up to here (see ce_rows_kernel); global accesses wait below
    griddep_launch_dependents();
    griddep_wait();
    // the first 32 labels fetched together, so no producer waits on one round trip per row
    const int64_t n_lab0 = min(n_it, static_cast<int64_t>(32));
    if (warp == 0 && lane < n_lab0) s_lab[lane] = __ldg(p.labels + cid + lane * ncl);
    __syncthreads();

    int64_t lab_lim = n_lab0;  // s_lab[0, lab_lim) holds labels
    auto label_of = [&](int64_t it) -> int64_t {
        return it < lab_lim ? s_lab[it] : __ldg(p.labels + cid + it * ncl);
    };
    bool aborted = false;
    auto check_abort = [&]() {
        if (!aborted && *reinterpret_cast<volatile int*>(&s_abort)) aborted = true;
    };

    // ---- producers.  The chunk sequence is: for every valid row, its chunks
    // for pass 1, then (fused) the same chunks again for pass 2; chunk k goes to
    // stage k % S.  Lane 0 of every warp walks this sequence S chunks ahead of
    // its own consumption, and the warp that releases chunk k last (a shared
    // counter per stage) issues chunk k + S into the freed stage: a stage is
    // refilled as soon as the slowest warp holds its chunk, and no thread ever
    // waits to issue.  Warp 0 issues the first S chunks.
    int64_t p_it = -1;          // row iteration of the cursor's chunk
    int p_pass = 0, p_chunk = 0, p_nchunk = 0;
    const char* p_src = nullptr;
    int64_t p_nb = 0;
    bool p_has = false;         // the cursor is on a chunk
    auto advance = [&]() {      // move the cursor to the next chunk
        if (p_has && !(p_pass == PASSES - 1 && p_chunk == p_nchunk - 1)) {
            if (p_chunk == p_nchunk - 1) {
                ++p_pass;
                p_chunk = 0;
            } else {
                ++p_chunk;
            }
            return;
        }
        p_has = false;
        for (int64_t it = p_it + 1; it < n_it; ++it) {
            if (!label_valid(label_of(it), p)) continue;
            const char* rowp = p.x + (cid + it * ncl) * row_bytes;
            const RowGeom gm = row_geom<ES>(rowp, p.V);
            const int nch = static_cast<int>((gm.nb + CHUNK - 1) / CHUNK);
            if (nch == 0) continue;  // scalars only: nothing to stream
            p_it = it;
            p_src = rowp + static_cast<int64_t>(gm.h) * ES;
            p_nb = gm.nb;
            p_nchunk = nch;
            p_pass = 0;
            p_chunk = 0;
            p_has = true;
            return;
        }
        p_it = n_it;
    };
    auto issue = [&](uint32_t st) {  // the cursor's chunk into stage st
        // test hook: the first load of one row is never made, so its stage never completes
        if (p_chunk == 0 && p_pass == 0 && p.skip_load_row == cid + p_it * ncl) return;
        const int64_t c0 = static_cast<int64_t>(p_chunk) * CHUNK;
        const uint32_t bytes = static_cast<uint32_t>(std::min<int64_t>(CHUNK, p_nb - c0)) * 16u;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&full[st], bytes);
        unsigned char* dst = smem + static_cast<size_t>(st) * p.stage_bytes;
        const int hint = p.l2_hint;
        if (hint == 0 || (hint == 2 && p_pass == 0)) {
            for (uint32_t off = 0; off < bytes; off += kBulkChunk)
                bulk_g2s(dst + off, p_src + c0 * 16 + off, min(kBulkChunk, bytes - off), &full[st]);
        } else {
            // pass 1 keeps the row in L2 for pass 2; pass 2 lets it go
            const uint64_t pol = p_pass == 0 ? l2_policy_evict_last() : l2_policy_evict_first();
            for (uint32_t off = 0; off < bytes; off += kBulkChunk)
                bulk_g2s_hint(dst + off, p_src + c0 * 16 + off, min(kBulkChunk, bytes - off), &full[st], pol);
        }
        ++s_iss[st];  // one issuer per stage at a time: the release protocol orders them
    };
    // One chunk's copy first, then the label reads (which would otherwise queue behind
    // every CTA's first S chunks of data), then the remaining S - 1 copies.
    uint32_t k_init = 0;
    if (lane == 0) {
        advance();
        if (p_has) {
            if (warp == 0) issue(0);
            advance();
            k_init = 1;
        }
    }

    int n_valid = 0, n_bad = 0;
    count_labels(p.count_labels, p.count_N, p.V, p.ignore_index, iscratch, n_valid, n_bad);
    const float D = row_denominator(p, n_valid);
    const float scale = p.g / D;
    for (int64_t it = tid; it < n_it && it < kLabCache; it += THREADS) s_lab[it] = __ldg(p.labels + cid + it * ncl);
    __syncthreads();
    lab_lim = kLabCache;
    if (lane == 0) {
        for (uint32_t k = k_init; k < S && p_has; ++k) {
            if (warp == 0) issue(k);
            advance();
        }
    }

    // For scale > 0 the scale is folded into the exponent; otherwise multiplied.
    const bool mul = !(scale > 0.f);
    const float log2_scale = mul ? 0.f : log2f(scale);

    uint32_t c_v = 0;  // chunks consumed
    uint32_t n_rows = 0;
    const uint4 pad = RowMath<ES>::pad();

    // Wait for the next chunk, move it into registers (-inf past its end) and
    // release its stage; the last warp to release it refills it.
    auto take_chunk = [&](int nl, uint4 (&v)[VPT]) {
        const uint32_t n = c_v, st = n % S;
        ++c_v;
        check_abort();
        if (!aborted && !mbar_wait_bounded(&full[st], (n / S) & 1u, p.wait_ns)) {
            s_abort = 1;
            aborted = true;
        }
        const uint4* sb = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(st) * p.stage_bytes);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int lv = tid + i * THREADS;
            v[i] = lv < nl ? sb[lv] : pad;
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();  // this warp's reads of the stage come before its release
            const unsigned prior = atomicAdd(&s_rel[st], 1u);
            if (prior % WARPS == WARPS - 1) {  // the last warp: every read is done
                __threadfence_block();
                check_abort();
                if (p_has && !aborted) issue(st);
            }
            advance();  // the cursor stays S chunks ahead of consumption
        }
    };

    for (int64_t it = 0; it < n_it; ++it) {
        const int64_t row = cid + it * ncl;
        const int64_t y = label_of(it);
        const char* rowp = p.x + row * row_bytes;
        const RowGeom gm = row_geom<ES>(rowp, p.V);
        const int nchunk = static_cast<int>((gm.nb + CHUNK - 1) / CHUNK);
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

        // Who owns the label column: the thread holding the head or tail scalar it
        // falls in, or the thread whose vector of chunk own_chunk contains it.  The
        // owner reads x_y straight from memory (one 32-byte sector per row) and,
        // after storing its vector, overwrites the label's gradient element.
        int own_chunk = -1, own_sc = -1;
        if (y < gm.h) {
            if (tid == 0) own_sc = static_cast<int>(y);
        } else if (y < tail_col) {
            const int64_t ly = y - gm.h;
            const int64_t lvec = ly / EPV;
            const int lv = static_cast<int>(lvec % CHUNK);
            if (lv % THREADS == tid) own_chunk = static_cast<int>(lvec / CHUNK);
        } else if (tid == 32) {
            own_sc = static_cast<int>(y - tail_col);
        }

        // ---- pass 1: running (max, sum) per thread, max shared by the warp
        float M = kNegInf, s = 0.f, x_y = 0.f;
        if (own_chunk >= 0) x_y = load_scalar<ES>(rowp + y * ES);
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
            M = warp_max_redux(xm);
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
            const int nl = static_cast<int>(std::min<int64_t>(CHUNK, gm.nb - static_cast<int64_t>(j) * CHUNK));
            uint4 v[VPT];
            take_chunk(nl, v);
            const float Mn = fmaxf(M, warp_max_redux(RowMath<ES>::template vmax<VPT>(v)));
            if (Mn != M) s *= ex2((M - Mn) * kLog2e);
            M = Mn;
            s += RowMath<ES>::template vsum<VPT>(v, M == kNegInf ? 0.f : M * kLog2e);
        }
        {
            const float sw = warp_sum(s);
            if (lane == 0) red_ms[rb][warp] = make_float2(M, sw);
        }
        __syncthreads();
        check_abort();
        const float2 pr = lane < WARPS ? red_ms[rb][lane] : make_float2(kNegInf, 0.f);
        const float Mr = warp_max_redux(pr.x);
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
                const int64_t cv0 = static_cast<int64_t>(j) * CHUNK;
                const int nl = static_cast<int>(std::min<int64_t>(CHUNK, gm.nb - cv0));
                uint4 v[VPT];
                take_chunk(nl, v);
                if (aborted) continue;
                uint4* dvc = dv + cv0;
                if (!mul) {
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        const int lv = tid + i * THREADS;
                        const uint4 o = RowMath<ES>::template vexp<false>(v[i], L2, C2, S2);
                        if (lv < nl) st_global_cs_v4(dvc + lv, o);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        const int lv = tid + i * THREADS;
                        const uint4 o = RowMath<ES>::template vexp<true>(v[i], L2, C2, S2);
                        if (lv < nl) st_global_cs_v4(dvc + lv, o);
                    }
                }
                if (j == own_chunk) {  // after this thread's own store of that vector
                    float d = ex2(fmaf(x_y, kLog2e, -c));
                    if (mul) d *= scale;
                    store_scalar<ES>(drow + y * ES, d - scale);
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
    __syncthreads();  // no warp issues any more
    if (tid == 0) {
        for (uint32_t st = 0; st < S; ++st)
            if (s_iss[st] > 0) (void)mbar_wait_bounded(&full[st], (s_iss[st] - 1u) & 1u, p.wait_ns);
    }
    rows_finish<THREADS>(p, aborted, n_valid, n_bad, &s_last, dred);
}

std::mutex g_long_mu;
std::map<std::pair<int, const void*>, bool> g_long_attr;  // (device, kernel): smem limit raised

template <int ES, bool GRAD, int THREADS, int VPT>
cudaError_t launch_long_typed(const CeRowParams& base, cudaStream_t stream) {
    const void* kern = reinterpret_cast<const void*>(&ce_rows_long_kernel<ES, GRAD, THREADS, VPT>);
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
    static const int forced_hint = [] {
        const char* e = std::getenv("FOAK_LONG_L2HINT");  // tuning override: 0, 1 or 2
        return e ? std::atoi(e) : -1;
    }();
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(device_sm_count(), base.N));
    // Rows held between the two passes: one per CTA.  Past half the 129 MB L2 the
    // second pass reads with evict_first, so the rows still waiting for it stay.
    const double in_flight = static_cast<double>(grid) * static_cast<double>(base.V) * ES;
    CeRowParams prm = base;
    prm.l2_hint = forced_hint >= 0 ? forced_hint : (in_flight > 64.0 * (1 << 20) ? 2 : 0);
    prm.k = 1;
    prm.per = THREADS * VPT;
    prm.stage_bytes = static_cast<uint32_t>(THREADS * VPT * 16);
    prm.stages = static_cast<int>(std::min<size_t>(kLongMaxStages, kSmemBudget / prm.stage_bytes));
    const size_t smem = static_cast<size_t>(prm.stages) * prm.stage_bytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr = pdl_attribute();
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ce_rows_long_kernel<ES, GRAD, THREADS, VPT>, prm);
}

template <int ES, bool GRAD>
cudaError_t launch_long_shape(const CeRowParams& base, cudaStream_t stream) {
    static const int threads = [] {
        const char* e = std::getenv("FOAK_LONG_THREADS");  // tuning override: 512, 768 or 1024
        return e ? std::atoi(e) : 0;
    }();
    if (threads == 768) return launch_long_typed<ES, GRAD, 768, 4>(base, stream);
    if (threads == 1024) return launch_long_typed<ES, GRAD, 1024, 4>(base, stream);
    return launch_long_typed<ES, GRAD, 512, 8>(base, stream);
}

}  // namespace

cudaError_t launch_ce_rows_long(bool grad, int elem_bytes, const CeRowParams& base, cudaStream_t stream) {
    if (elem_bytes == 2) return grad ? launch_long_shape<2, true>(base, stream) : launch_long_shape<2, false>(base, stream);
    return grad ? launch_long_shape<4, true>(base, stream) : launch_long_shape<4, false>(base, stream);
}

}  // namespace foak
