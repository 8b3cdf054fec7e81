// Row-wise cross-entropy (forward, and fused forward+backward in place) for rows
// of at most 64 KB that start on a 16-byte boundary and end on a whole vector --
// the Mistral, packed and chunked linear + CE workloads -- with the 16 warps of
// a CTA working independently instead of in step.  The forward call uses it for
// such rows (58.0 -> 56.3 us on the 4096 x 32000 bf16 batch); the fused sweep is
// faster on the CTA-in-step kernel of ce_rows.cu (95 against 104 us) and reaches
// this one only through the row-path test hook.
//
// One CTA per SM takes rows round-robin.  Warp w owns a 4 KB region of every row
// (vectors 256w .. 256w + 255; lane l holds vectors 256w + 32i + l, i < 8) and
// moves it through a ring of three 64 KB shared-memory stages by itself: it
// issues the bulk copy (TMA engine) of its region of a row, waits for the row's
// stage to fill, copies its region to registers and at once refills the region
// with the row three valid rows ahead.  The only thing the warps share per row is
// the log-sum-exp: each warp sends its (max, sum of exp) pair with st.async into
// a slot of an 8-row ring, completing bytes on that slot's mbarrier, and reads
// the 16 pairs one row later -- after it has formed its pair of the next row --
// so a warp almost never waits for the others, and the loads, exponentials and
// 16-byte streaming stores of different warps overlap instead of taking turns.
// The forward only needs a row's log-sum-exp for its outputs, so only the warp
// whose region holds the label reads the pairs and writes lse and the row term
// (51.1 -> 47.1 us on the Mistral batch against every warp merging them).
// The fused kernel then writes (exp(x - lse) - onehot) * g / D over the logits
// from the registers it kept; ignored rows are never read, only zero-filled.
// This is the one-pass row sweep of the FastCrossEntropyLoss kernel the FOAK
// pages describe (fms-acceleration PR #79, Description item 4), scheduled for
// sm_103a.
//
// Ring safety: a warp sends its pair of valid row k only after every warp issued
// its copy of row k, which each does right after taking row k - 3 into
// registers, i.e. after finishing row k - 5's log-sum-exp; with 8 pair slots no
// slot is overwritten before all warps have read it.
#include <algorithm>
#include <mutex>

#include "row_common.cuh"

namespace foak {

namespace {

constexpr int kWThreads = 512;
constexpr int kWWarps = kWThreads / 32;
constexpr int kWVpt = 8;                    // 16-byte vectors per lane and row
constexpr int kWRegion = 32 * kWVpt;        // vectors per warp region (4 KB)
constexpr int kWStages = 3;
constexpr int kWPairSlots = 8;
constexpr uint32_t kWStageBytes = kRowSliceVecMax * 16;  // 64 KB

// Bounded wait that also gives up as soon as another warp has recorded an abort;
// it spins on test_wait (measured: forward 57.8 -> 56.4 us against try_wait).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

}  // namespace

template <int ES, bool GRAD>
__global__ void __launch_bounds__(kWThreads, 1) ce_rows_warp_kernel(const CeRowParams p) {
    constexpr int EPV = 16 / ES;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t full[kWStages];
    __shared__ uint64_t rowdone[kWPairSlots];
    __shared__ float2 pairs[kWPairSlots][kWWarps];
    __shared__ int64_t s_lab[kLabCache];
    __shared__ int iscratch[2 * kWWarps];
    __shared__ DFloat dred[kWWarps];
    __shared__ volatile int s_abort;
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // rows, iterations and valid labels all fit 32 bits (the host checks N < 2^31)
    const int cid = static_cast<int>(blockIdx.x);
    const int ncl = static_cast<int>(gridDim.x);
    const int n_it = p.N > cid ? static_cast<int>((p.N - 1 - cid) / ncl + 1) : 0;
    const int64_t row_bytes = p.ld * ES;
    const int nl = static_cast<int>(p.V / EPV);                           // vectors per row
    const int r0 = warp * kWRegion;                                        // this warp's first vector
    const int nreg = max(0, min(static_cast<int>(kWRegion), nl - r0));    // its vectors in a row
    const uint32_t reg_bytes = static_cast<uint32_t>(nreg) * 16u;

    if (tid == 0) {
        for (int s = 0; s < kWStages; ++s) mbar_init(&full[s], kWWarps);
        for (int s = 0; s < kWPairSlots; ++s) mbar_init(&rowdone[s], 1);
        fence_mbar_init();
        s_abort = 0;
        s_last = 0;
    }
    // -inf in this lane's slots past the row (the copies never write there), every stage
    {
        const uint4 pad = RowMath<ES>::pad();
#pragma unroll
        for (int i = 0; i < kWVpt; ++i) {
            const int lv = r0 + 32 * i + lane;
            if (lv >= nl)
                for (int s = 0; s < kWStages; ++s)
                    reinterpret_cast<uint4*>(smem + static_cast<size_t>(s) * kWStageBytes)[lv] = pad;
        }
    }
    // shared memory only up to here: under a programmatic launch this overlaps the end
    // of the previous kernel, and every global access below waits for it
    griddep_launch_dependents();
    griddep_wait();
    // the first 32 labels fetched together, so no warp waits on one round trip per row
    const int n_lab0 = min(n_it, 32);
    if (warp == 0 && lane < n_lab0) s_lab[lane] = __ldg(p.labels + cid + lane * ncl);
    __syncthreads();

    // Producer state of this warp (lane 0): next row iteration to scan, valid rows issued.
    int q_it = 0;
    uint32_t q_v = 0;
    int lab_lim = n_lab0;  // s_lab[0, lab_lim) holds labels
    auto label_of = [&](int it) -> int64_t {
        return it < lab_lim ? s_lab[it] : __ldg(p.labels + cid + it * ncl);
    };
    auto is_valid = [&](int64_t y) { return y != p.ignore_index && y >= 0 && y < p.V; };
    // Copy this warp's region of the next valid row into its stage (lane 0).
    auto issue_next = [&]() {
        while (q_it < n_it) {
            const int row = cid + q_it * ncl;
            const int64_t y = label_of(q_it);
            ++q_it;
            if (!is_valid(y)) continue;
            const int st = static_cast<int>(q_v % kWStages);
            ++q_v;
            if (row == p.skip_load_row) return;  // test hook: this stage phase never completes
            mbar_arrive_expect_tx(&full[st], reg_bytes);
            if (reg_bytes)
                bulk_g2s(smem + static_cast<size_t>(st) * kWStageBytes + static_cast<size_t>(r0) * 16,
                         p.x + static_cast<int64_t>(row) * row_bytes + static_cast<int64_t>(r0) * 16, reg_bytes,
                         &full[st]);
            return;
        }
    };
    // One row's copies first, then the label reads (which would otherwise queue behind
    // every CTA's three rows of data), then the remaining copies.
    if (lane == 0) issue_next();

    // The forward needs the denominator only for the loss: when the call counts its own
    // labels, each CTA counts those of its rows on the way and the last CTA adds them up
    // (no read of all N labels by every CTA at start-up).  The fused sweep scales every
    // gradient by g / D, so it counts first.
    const bool late_count = !GRAD && p.count_labels == p.labels && p.count_N == p.N;
    int n_valid = 0, n_bad = 0;
    if (!late_count) count_labels(p.count_labels, p.count_N, p.V, p.ignore_index, iscratch, n_valid, n_bad);
    const float D = row_denominator(p, n_valid);
    const float scale = p.g / D;
    for (int it = n_lab0 + tid; it < n_it && it < kLabCache; it += kWThreads) s_lab[it] = __ldg(p.labels + cid + it * ncl);
    __syncthreads();
    lab_lim = kLabCache;
    if (lane == 0)
        for (int s = 1; s < kWStages; ++s) issue_next();

    // Gradient constants: for scale > 0 the scale is folded into the exponent,
    // 2^(x*log2e - lse2 + log2(scale)); otherwise the exponential is multiplied by it.
    const bool mul = !(scale > 0.f);
    const float log2_scale = mul ? 0.f : log2f(scale);
    const uint32_t my_rank = cluster_ctarank();

    bool aborted = false;
    uint32_t c_v = 0;   // valid rows taken into registers
    uint32_t c_ok = 0;  // valid rows whose copy was seen complete (a prefix)

    // The row whose log-sum-exp is still to be formed (one behind the current).
    uint4 va[kWVpt], vb[kWVpt];
    bool pend = false;
    int pend_row = 0, pend_y = 0;
    uint32_t pend_j = 0;
    bool pend_own = false;
    bool pend_own_w = false;  // the label's vector is in this warp's region
    float pend_xy = 0.f;

    auto give_up = [&]() {
        aborted = true;
        s_abort = 1;
    };

    // Log-sum-exp of the pending row from the 16 pairs, its outputs and (fused) its gradient.
    auto finish_row = [&](const uint4 (&v)[kWVpt]) {
        // forward: only the warp holding the label needs the row's log-sum-exp
        if constexpr (!GRAD) {
            if (!pend_own_w) return;
        }
        const uint32_t slot = pend_j % kWPairSlots;
        if (!aborted && !wait_or_abort(&rowdone[slot], (pend_j / kWPairSlots) & 1u, p.wait_ns, &s_abort)) give_up();
        const float2 pr = lane < kWWarps ? pairs[slot][lane] : make_float2(kNegInf, 0.f);
        const float M = warp_max_redux(pr.x);
        const float S = warp_sum(pr.x == kNegInf ? 0.f : pr.y * ex2((pr.x - M) * kLog2e));
        const float lse2 = fmaf(M, kLog2e, lg2(S));
        const float lse = lse2 * kLn2;
        if (aborted) return;
        if (pend_own) p.row_loss[pend_row] = lse - pend_xy;
        if ((GRAD ? tid == 0 : lane == 0) && p.lse) p.lse[pend_row] = lse;
        if constexpr (GRAD) {
            const float c = lse2 - log2_scale;
            const f32x2_t L2 = f2_pack(kLog2e, kLog2e), C2 = f2_pack(-c, -c), S2 = f2_pack(scale, scale);
            char* drow = p.dx + static_cast<int64_t>(pend_row) * row_bytes;
            uint4* dv = reinterpret_cast<uint4*>(drow);
            if (!mul) {
#pragma unroll
                for (int i = 0; i < kWVpt; ++i) {
                    const int lv = r0 + 32 * i + lane;
                    const uint4 o = RowMath<ES>::template vexp<false>(v[i], L2, C2, S2);
                    if (lv < nl) st_global_cs_v4(dv + lv, o);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kWVpt; ++i) {
                    const int lv = r0 + 32 * i + lane;
                    const uint4 o = RowMath<ES>::template vexp<true>(v[i], L2, C2, S2);
                    if (lv < nl) st_global_cs_v4(dv + lv, o);
                }
            }
            if (pend_own) {  // the label's element, after this thread's store of its vector
                float d = ex2(fmaf(pend_xy, kLog2e, -c));
                if (mul) d *= scale;
                store_scalar<ES>(drow + static_cast<int64_t>(pend_y) * ES, d - scale);
            }
        }
    };

    for (int it = 0; it < n_it; ++it) {
        const int row = cid + it * ncl;
        const int64_t y = label_of(it);
        if (late_count && tid == 0) {
            if (is_valid(y)) ++n_valid;
            else if (y != p.ignore_index) ++n_bad;
        }
        if (!is_valid(y)) {
            if constexpr (GRAD) {
                if (!aborted) {
                    uint4* dv = reinterpret_cast<uint4*>(p.dx + static_cast<int64_t>(row) * row_bytes);
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int i = 0; i < kWVpt; ++i) {
                        const int lv = r0 + 32 * i + lane;
                        if (lv < nl) st_global_cs_v4(dv + lv, z);
                    }
                }
            }
            if (tid == 0) {
                p.row_loss[row] = 0.f;
                if (p.lse) p.lse[row] = 0.f;
            }
            continue;
        }
        // This lane owns the label column when the label's vector is one of its slots;
        // it reads x_y from memory now, so the load overlaps the wait and the arithmetic.
        const int yv = static_cast<int>(y / EPV);
        const bool own_w = yv >= r0 && yv < r0 + kWRegion;
        const bool own = own_w && ((yv - r0) & 31) == lane;
        float x_y = 0.f;
        if (own) x_y = load_scalar<ES>(p.x + static_cast<int64_t>(row) * row_bytes + y * ES);

        const uint32_t j = c_v++;
        const int st = static_cast<int>(j % kWStages);
        if (!aborted) {
            if (wait_or_abort(&full[st], (j / kWStages) & 1u, p.wait_ns, &s_abort)) c_ok = c_v;
            else give_up();
        }
        const uint4* sb = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(st) * kWStageBytes);
#pragma unroll
        for (int i = 0; i < kWVpt; ++i) vb[i] = sb[r0 + 32 * i + lane];
        float m = RowMath<ES>::template vmax<kWVpt>(vb);
        m = warp_max_redux(m);  // every slot is in registers now: the region may be refilled
        if (lane == 0 && !aborted) issue_next();
        const float mb = m == kNegInf ? 0.f : m * kLog2e;
        const float sum = warp_sum(RowMath<ES>::template vsum<kWVpt>(vb, mb));
        if (lane == 0 && !aborted) {
            const uint32_t slot = j % kWPairSlots;
            if (warp == 0) mbar_arrive_expect_tx(&rowdone[slot], 8u * kWWarps);
            st_async_f2(mapa_u32(&pairs[slot][warp], my_rank), m, sum, mapa_u32(&rowdone[slot], my_rank));
        }
        // the previous row's log-sum-exp (its pairs have had a whole row's time to arrive)
        if (pend) finish_row(va);
#pragma unroll
        for (int i = 0; i < kWVpt; ++i) va[i] = vb[i];
        pend = true;
        pend_row = row;
        pend_y = static_cast<int>(y);
        pend_j = j;
        pend_own = own;
        pend_own_w = own_w;
        pend_xy = x_y;
    }
    if (pend) finish_row(va);

    // Copies still in flight exist only after an abort: let the ones this warp issued land.
    if (lane == 0) {
        for (uint32_t k = c_ok; k < q_v; ++k)
            (void)mbar_wait_bounded(&full[k % kWStages], (k / kWStages) & 1u, p.wait_ns);
    }
    __syncthreads();  // an abort seen by any warp is reported
    rows_finish<kWThreads>(p, aborted || s_abort != 0, n_valid, n_bad, &s_last, dred, late_count);
}

// ------------------------------------------------------------------ host side

namespace {
std::mutex g_wmu;
bool g_wattr[64][4] = {};
}  // namespace

bool ce_rows_warp_fits(int elem_bytes, int64_t V) {
    return V >= 1 && V * elem_bytes <= static_cast<int64_t>(kWStageBytes) && (V * elem_bytes) % 16 == 0;
}

template <int ES, bool GRAD>
static cudaError_t launch_warp_typed(const CeRowParams& prm, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const size_t smem = static_cast<size_t>(kWStages) * kWStageBytes;
    const int ki = (ES == 2 ? 0 : 2) + (GRAD ? 1 : 0);
    {
        std::lock_guard<std::mutex> lock(g_wmu);
        if (!g_wattr[dev][ki]) {
            e = cudaFuncSetAttribute(ce_rows_warp_kernel<ES, GRAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            g_wattr[dev][ki] = true;
        }
    }
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(device_sm_count(), prm.N));
    // a cluster of one CTA, explicitly: the pairs travel by st.async into the CTA's own shared memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kWThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, ce_rows_warp_kernel<ES, GRAD>, prm);
}

cudaError_t launch_ce_rows_warp(bool grad, int elem_bytes, const CeRowParams& prm, cudaStream_t stream) {
    if (elem_bytes == 2) return grad ? launch_warp_typed<2, true>(prm, stream) : launch_warp_typed<2, false>(prm, stream);
    return grad ? launch_warp_typed<4, true>(prm, stream) : launch_warp_typed<4, false>(prm, stream);
}

}  // namespace foak
