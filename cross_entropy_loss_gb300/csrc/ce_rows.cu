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
// N = 8192, an L2-resident read), and the mean loss is reduced (a double-float
// sum in a fixed order) by whichever CTA finishes last.
#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "row_common.cuh"

namespace foak {

// AL: every row starts on a 16-byte boundary and V * ES is a multiple of 16, so
// rows have no scalar head or tail and every row's slice has the same length;
// the stage slots past it are filled with -inf once and loaded unconditionally.
template <int ES, bool GRAD, int THREADS, bool AL>
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
    __shared__ DFloat dred[kRowWarps];
    __shared__ int s_abort, s_last;
    // Single-CTA rows: the batch's valid rows from row tail0 on, in row order (the
    // same list in every CTA), handed out one at a time through the workspace
    // header's counter, and the row and label whose copy went into each stage.
    constexpr int kTail = THREADS >= 512 ? kTailMax : 1;
    __shared__ int2 s_tail[kTail];  // (row, label): labels of valid rows fit 32 bits
    __shared__ int s_ntail;
    __shared__ int s_scan[kRowWarps];  // the tail scan's warp totals (count_labels has its own scratch)
    __shared__ int s_qrow[kRowMaxStages];
    __shared__ int64_t s_qlab[kRowMaxStages];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.k;
    const int rank = K > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int64_t cid = K > 1 ? cluster_id_x() : blockIdx.x;
    const int64_t ncl = K > 1 ? cluster_count_x() : gridDim.x;
    const int64_t n_it = p.N > cid ? (p.N - 1 - cid) / ncl + 1 : 0;
    // With a tail, this CTA's round-robin rows are those below tail0; the rest are
    // shared.  Whether the call takes a tail is decided once the labels are counted
    // (below); until then only rows that are round-robin either way are touched.
    const bool dyn_ok = K == 1 && kTail > 1 && p.tail_rounds >= 0;
    const int64_t tail_lo = dyn_ok ? static_cast<int64_t>(p.tail_rounds) * ncl : p.N;
    const int64_t n_stat_lo = tail_lo > cid ? (tail_lo - 1 - cid) / ncl + 1 : 0;
    bool dyn = dyn_ok;
    int64_t tail0 = tail_lo;
    int64_t n_stat = n_stat_lo;
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
    if constexpr (AL) {
        // -inf in every stage slot past this CTA's slice (the copies never write there)
        int64_t nl0 = p.V / EPV - v0;
        nl0 = nl0 < 0 ? 0 : (nl0 > p.per ? p.per : nl0);
        const uint4 pad = RowMath<ES>::pad();
        for (int s = 0; s < p.stages; ++s) {
            uint4* sb = reinterpret_cast<uint4*>(smem + static_cast<size_t>(s) * p.stage_bytes);
            for (int i = static_cast<int>(nl0) + tid; i < VPT * kRowThreads; i += kRowThreads) sb[i] = pad;
        }
    }
    __syncthreads();
    if (K > 1) cluster_sync();  // every CTA's exchange barriers exist before the first st.async
    // Up to here only shared memory was touched: under a programmatic launch this
    // set-up overlaps the end of the previous kernel, and everything below waits for it.
    griddep_launch_dependents();
    griddep_wait();

    // Producer state (thread 0): next row iteration to look at, valid rows issued.
    int64_t p_it = 0;
    uint32_t p_v = 0;
    int64_t lab_lim = 0;  // labels s_lab[0, lab_lim) are valid for this thread
    auto label_of = [&](int64_t it) -> int64_t {
        return it < lab_lim ? s_lab[it] : __ldg(p.labels + cid + it * ncl);
    };
    // Fused kernel: the next load is found (label scan, address, size) before
    // the row's barrier and only issued after it, so thread 0's warp leaves the
    // barrier with little extra work and does not hold up the next one.
    const char* q_src = nullptr;
    uint32_t q_bytes = 0;
    int64_t q_row = 0, q_lab = 0;
    int q_state = 0;  // 0 nothing prepared, 1 a load, 2 a skipped load (test hook), 3 no rows left
    // Tail claims: the counter is bumped one claim ahead, so the atomic's latency is
    // hidden behind a row instead of delaying thread 0 at a row barrier.
    unsigned claim = 0;
    bool claim_out = false;
    bool ended = false;  // the end of the row sequence has been marked in s_qrow
    auto claim_ahead = [&]() {
        if (dyn && !claim_out) {
            claim = atomicAdd(&p.ws->next, 1u);
            claim_out = true;
        }
    };
    // The next valid row of this CTA: its round-robin rows, then claimed tail rows.
    auto next_row = [&](int64_t& row, int64_t& y) -> bool {
        while (p_it < n_stat) {
            row = cid + p_it * ncl;
            y = label_of(p_it);
            ++p_it;
            if (dyn && p_it + 1 >= n_stat) claim_ahead();
            if (y == p.ignore_index || y < 0 || y >= p.V) continue;
            return true;
        }
        if (!dyn) return false;
        claim_ahead();
        const unsigned k = claim;
        claim_out = false;
        if (k >= static_cast<unsigned>(s_ntail)) return false;
        const int2 e = s_tail[k];
        row = e.x;
        y = e.y;
        claim_ahead();  // the next claim, already on its way
        return true;
    };
    auto prepare = [&]() {
        if (q_state != 0) return;
        int64_t row, y;
        if (!next_row(row, y)) {
            q_state = 3;
            return;
        }
        q_row = row;
        q_lab = y;
        if (row == p.skip_load_row) {  // test hook: the stage's barrier is never completed
            q_state = 2;
            return;
        }
        const char* rowp = p.x + row * row_bytes;
        const RowGeom gm = AL ? RowGeom{0, p.V / EPV, 0} : row_geom<ES>(rowp, p.V);
        int64_t nl = gm.nb - v0;
        nl = nl < 0 ? 0 : (nl > p.per ? p.per : nl);
        q_bytes = static_cast<uint32_t>(nl) * 16u;
        q_src = rowp + static_cast<int64_t>(gm.h) * ES + v0 * 16;
        q_state = 1;
    };
    auto fire = [&]() {
        const int st = static_cast<int>(p_v % static_cast<uint32_t>(p.stages));
        if (q_state == 1) {
            uint64_t* bar = &bars[st];
            mbar_arrive_expect_tx(bar, q_bytes);
            unsigned char* dst = smem + static_cast<size_t>(st) * p.stage_bytes;
            for (uint32_t off = 0; off < q_bytes; off += kBulkChunk)
                bulk_g2s(dst + off, q_src + off, min(kBulkChunk, q_bytes - off), bar);
        }
        if (q_state == 1 || q_state == 2) {
            s_qrow[st] = static_cast<int>(q_row);
            s_qlab[st] = q_lab;
            ++p_v;
            q_state = 0;
        } else if (q_state == 3 && dyn && !ended) {
            s_qrow[st] = -1;  // the consumers stop at this stage
            ended = true;
        }
    };
    auto issue_next = [&]() {
        prepare();
        fire();
    };
    // Start-up order matters: every CTA reads all N labels (the count) and its own
    // rows' labels, and if the first copies of all CTAs (three 64 KB rows each) went
    // out first, those small reads would queue behind ~29 MB of row data.  So warp 0
    // fetches the first 32 labels together, thread 0 issues the first row's copy,
    // all label reads follow, and then the remaining copies.  A copy that would need
    // a claimed tail row waits until the tail list exists.
    const int64_t n_lab0 = min(n_stat_lo, static_cast<int64_t>(32));
    if (warp == 0) {
        if (lane < n_lab0) s_lab[lane] = __ldg(p.labels + cid + lane * ncl);
        __syncwarp();
        lab_lim = n_lab0;
    }
    int n_early = 0;
    if (tid == 0) {
        bool have = !dyn;
        for (int64_t i = p_it; i < n_stat && !have; ++i) {
            const int64_t y = label_of(i);
            have = y != p.ignore_index && y >= 0 && y < p.V;
        }
        if (have) {
            issue_next();
            n_early = 1;
        }
    }

    int n_valid = 0, n_bad = 0;
    count_labels(p.count_labels, p.count_N, p.V, p.ignore_index, iscratch, n_valid, n_bad);
    const float D = row_denominator(p, n_valid);
    const float scale = p.g / D;
    // The shared tail pays only when the round-robin split is uneven, i.e. when many
    // rows are ignored (they take no load): measured on 8192-row padding-free batches
    // (45% ignored) 148 -> 141 us, while on the Mistral batch (0.1% ignored) the tail's
    // extra start-up costs 3 us.  Every CTA counts the same labels, so all agree; a
    // call whose count covers other rows than its own (a chunk of a larger batch) keeps
    // the round-robin split.
    if (dyn_ok && (p.count_labels != p.labels || p.count_N != p.N || (p.N - n_valid) * static_cast<int64_t>(kTailIgnoredDiv) < p.N)) {
        dyn = false;
        tail0 = p.N;
        n_stat = n_it;
    }
    // Labels of this CTA's rows (round-robin ones, then its share of the tail: rows
    // tail0 + cid + j * ncl, which it zero-fills when they are ignored); warp 0
    // already holds the first n_lab0.
    const int64_t n_mine = dyn ? (p.N > tail0 + cid ? (p.N - 1 - tail0 - cid) / ncl + 1 : 0) : 0;
    for (int64_t it = n_lab0 + tid; it < n_stat + n_mine && it < kLabCache; it += blockDim.x)
        s_lab[it] = __ldg(p.labels + (it < n_stat ? cid + it * ncl : tail0 + cid + (it - n_stat) * ncl));
    // The shared tail's valid rows, in row order: every thread counts a block of
    // labels, a CTA scan gives each block its place, and each block writes its rows.
    if (dyn) {
        const int64_t T = p.N - tail0;  // at most kTailMax (the host sizes tail_rounds so)
        constexpr int kPer = (kTail + kRowThreads - 1) / kRowThreads;
        const int per_t = static_cast<int>((T + kRowThreads - 1) / kRowThreads);
        const int64_t b0 = tail0 + static_cast<int64_t>(tid) * per_t;
        int64_t yb[kPer];  // this thread's block of labels, loaded together
        int cnt = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            yb[k] = (k < per_t && b0 + k < p.N) ? __ldg(p.labels + b0 + k) : p.ignore_index;
            cnt += (yb[k] != p.ignore_index && yb[k] >= 0 && yb[k] < p.V) ? 1 : 0;
        }
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) s_scan[warp] = incl;
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w) base += s_scan[w];
        int pos = base + incl - cnt;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            if (yb[k] != p.ignore_index && yb[k] >= 0 && yb[k] < p.V)
                s_tail[pos++] = make_int2(static_cast<int>(b0 + k), static_cast<int>(yb[k]));
        }
        if (tid == kRowThreads - 1) s_ntail = base + incl;
    }
    __syncthreads();
    lab_lim = kLabCache;
    // the remaining copies; the barrier publishes what thread 0 recorded for them
    if (tid == 0)
        for (int s = n_early; s < p.stages; ++s) issue_next();
    __syncthreads();

    // Gradient constants: for scale > 0 the scale is folded into the exponent,
    // 2^(x*log2e - lse2 + log2(scale)); otherwise the exponential is multiplied by it.
    const bool mul = !(scale > 0.f);
    const float log2_scale = mul ? 0.f : log2f(scale);

    int c_st = 0;          // stage of the next valid row
    uint32_t c_par = 0;    // its phase parity
    uint32_t c_v = 0;      // valid rows consumed
    uint32_t c_ok = 0;     // valid rows whose load was seen complete (a prefix)
    bool aborted = false;
    auto do_row = [&](const int64_t row, const int64_t y) {
        const bool valid = y != p.ignore_index && y >= 0 && y < p.V;
        const char* rowp = p.x + row * row_bytes;
        const RowGeom gm = AL ? RowGeom{0, p.V / EPV, 0} : row_geom<ES>(rowp, p.V);
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
            return;
        }

        // Who owns the label column: the thread holding the head or tail scalar it
        // falls in, or the thread whose vector contains it (no division: kRowThreads
        // is a power of 2).  A vector owner reads x_y from memory now, so the load
        // overlaps the row's wait and arithmetic, and later patches the label's
        // gradient element with a scalar store: no per-vector label work.
        bool own_vec = false;
        int own_sc = -1;
        if (y < gm.h) {
            if (rank == 0 && tid == 0) own_sc = static_cast<int>(y);
        } else if (y < tail_col) {
            const int64_t lv = (y - gm.h) / EPV - v0;
            own_vec = lv >= 0 && lv < p.per && (static_cast<int>(lv) & (kRowThreads - 1)) == tid;
        } else if (rank == K - 1 && tid == tail_tid) {
            own_sc = static_cast<int>(y - tail_col);
        }
        float x_y = 0.f;
        if (own_vec) x_y = load_scalar<ES>(rowp + y * ES);

        const int st = c_st;
        const uint32_t par = c_par;
        if (++c_st == p.stages) {
            c_st = 0;
            c_par ^= 1u;
        }
        ++c_v;
        if (!aborted) {
            if (mbar_wait_bounded(&bars[st], par, p.wait_ns)) c_ok = c_v;
            else s_abort = 1;
        }

        // Slice -> registers (vectors past the slice hold -inf); scalars from global memory.
        uint4 v[VPT];
        const uint4* sb = reinterpret_cast<const uint4*>(smem + static_cast<size_t>(st) * p.stage_bytes);
        const uint4 pad = RowMath<ES>::pad();
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int lv = tid + i * kRowThreads;
            v[i] = (AL || lv < nl) ? sb[lv] : pad;
        }
        if (GRAD && tid == 0 && !aborted) prepare();  // measured: the forward sweep runs faster without
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
        m = GRAD ? warp_max(m) : warp_max_redux(m);  // measured: shuffles for the fused kernel
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
            issue_next();  // fused: only fires what was prepared before the barrier
        }
        const float2 pr = lane < kRowWarps ? red_ms[rb][lane] : make_float2(kNegInf, 0.f);
        float M = GRAD ? warp_max(pr.x) : warp_max_redux(pr.x);
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

        if (own_sc >= 0) {
#pragma unroll
            for (int s = 0; s < kMaxScalars; ++s)
                if (s == own_sc) x_y = xs[s];
        }
        if ((own_vec || own_sc >= 0) && !aborted) p.row_loss[row] = lse - x_y;

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
                        const uint4 o = RowMath<ES>::template vexp<false>(v[i], L2, C2, S2);
                        if (lv < nl) st_global_cs_v4(dv + lv, o);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VPT; ++i) {
                        const int lv = tid + i * kRowThreads;
                        const uint4 o = RowMath<ES>::template vexp<true>(v[i], L2, C2, S2);
                        if (lv < nl) st_global_cs_v4(dv + lv, o);
                    }
                }
                if (own_vec) {  // the label's element, after this thread's store of its vector
                    float d = ex2(fmaf(x_y, kLog2e, -c));
                    if (mul) d *= scale;
                    store_scalar<ES>(drow + y * ES, d - scale);
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
    };

    // One loop, one copy of the row code: this CTA's round-robin rows; then its share
    // of the tail's ignored rows (only written: +0.0 and zero row terms); then the
    // tail's valid rows it claimed, in the order their copies were issued, until the
    // stage marked as the end (written by thread 0 at least one row barrier before
    // any thread reads it).
    for (int64_t it = 0;; ++it) {
        int64_t row, y;
        if (it < n_stat) {
            row = cid + it * ncl;
            y = label_of(it);
        } else if (it < n_stat + n_mine) {
            row = tail0 + cid + (it - n_stat) * ncl;
            y = it < kLabCache ? s_lab[it] : __ldg(p.labels + row);
            if (y != p.ignore_index && y >= 0 && y < p.V) continue;  // a tail row for the claims
        } else {
            if (!dyn || aborted) break;
            row = s_qrow[c_st];
            if (row < 0) break;
            y = s_qlab[c_st];
        }
        do_row(row, y);
    }

    // Loads still in flight exist only after an abort: those issued past the
    // last one seen complete may still be landing; let them land first.
    if (tid == 0) {
        const uint32_t S = static_cast<uint32_t>(p.stages);
        for (uint32_t k = c_ok; k < p_v; ++k) (void)mbar_wait_bounded(&bars[k % S], (k / S) & 1u, p.wait_ns);
    }
    if (K > 1) cluster_sync();  // no CTA leaves while a peer may still send it a pair

    rows_finish<THREADS>(p, aborted, n_valid, n_bad, &s_last, dred);
}

// ------------------------------------------------------------------ host side

int64_t ce_rows_max_vocab(int elem_bytes) {
    // rows past the one-pass plans (8 CTAs x 64 KB) are streamed twice by one CTA,
    // whose chunk and column indexes are 32-bit
    (void)elem_bytes;
    return 0x7fffffffLL;
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

bool plan_needs_cluster(int ES, int64_t V) {
    Plan one;
    return !plan_with(ES, V, 512, kRowSliceVecMax, kSmemBudget, &one) || one.k > 1;
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

template <int ES, bool GRAD, int THREADS, bool AL>
cudaError_t launch_typed(const CeRowParams& base, const Plan& pl, cudaStream_t stream) {
    const void* kern = reinterpret_cast<const void*>(&ce_rows_kernel<ES, GRAD, THREADS, AL>);
    int ncl = 0;
    cudaError_t e = resident_clusters(kern, THREADS, pl.k, pl.smem, &ncl);
    if (e != cudaSuccess) return e;
    const int64_t want = std::max<int64_t>(1, std::min<int64_t>(ncl, base.N));
    CeRowParams prm = base;
    // Single-CTA rows: about 80% of the rows go round-robin and the valid rows of the
    // rest are handed out at run time, so the CTAs (whose speed and share of valid
    // rows differ) finish together; the shared tail is at most kTailMax rows.
    prm.tail_rounds = -1;
    if (pl.k == 1 && THREADS >= 512) {
        const int64_t rounds = base.N / want;
        int64_t tr = rounds * 8 / 10;
        tr = std::max<int64_t>(tr, (base.N - kTailMax + want - 1) / want);
        prm.tail_rounds = static_cast<int>(std::min<int64_t>(std::max<int64_t>(tr, 0), rounds));
    }
    prm.k = pl.k;
    prm.per = pl.per;
    prm.stages = pl.stages;
    prm.stage_bytes = pl.stage_bytes;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want * pl.k), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(pl.k);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();  // the shared-memory set-up may overlap the previous kernel's end
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, ce_rows_kernel<ES, GRAD, THREADS, AL>, prm);
}

// Aligned rows on one CTA each take the AL kernel, whose stages hold a full
// slice (THREADS x VPT vectors) so the pad slots exist.
template <int ES, bool GRAD>
cudaError_t launch_vpt(const CeRowParams& base, const Plan& pl, cudaStream_t stream, bool aligned) {
    if (pl.threads == 256) return launch_typed<ES, GRAD, 256, false>(base, pl, stream);
    if (aligned && pl.k == 1) {
        // 512 x 8 by default; 1024 x 4 (64 registers) as a tuning override
        static const int forced = [] {
            const char* e = std::getenv("FOAK_ROW_THREADS");
            return e ? std::atoi(e) : 0;
        }();
        const int threads = forced == 1024 ? 1024 : 512;
        Plan full = pl;
        full.stage_bytes = kRowSliceVecMax * 16;
        full.stages = static_cast<int>(std::min<size_t>(kRowMaxStages, kSmemBudget / full.stage_bytes));
        full.smem = static_cast<size_t>(full.stages) * full.stage_bytes;
        return threads == 1024 ? launch_typed<ES, GRAD, 1024, true>(base, full, stream)
                               : launch_typed<ES, GRAD, 512, true>(base, full, stream);
    }
    return pl.threads == 1024 ? launch_typed<ES, GRAD, 1024, false>(base, pl, stream)
                              : launch_typed<ES, GRAD, 512, false>(base, pl, stream);
}

}  // namespace

cudaError_t launch_ce_rows(bool grad, int elem_bytes, const void* x, void* dx, int64_t ld,
                           const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index, float g,
                           float denom, float* loss, float* lse, float* row_loss, int32_t* n_valid,
                           int32_t* err, CeWsHeader* ws, cudaStream_t stream, const int64_t* count_labels,
                           int64_t count_N, const int64_t* denom_dev) {
    Plan pl;
    const bool planned = plan_rows(elem_bytes, V, &pl);  // false past the one-pass plans' reach
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
    prm.denom_dev = denom_dev;
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
    // Rows longer than one 512-thread CTA's slice are streamed twice by one CTA
    // (every SM busy, no cluster exchange) unless the one-pass cluster kernel is asked
    // for; rows too long for any one-pass plan always are.
    const int hook = test_row_path();
    const bool warp_ok = hook != 1 && hook != 2;  // 3 asks for the independent-warp kernel, like 0
    const int path = hook == 3 ? 0 : hook;
    if (!planned || path == 2 || (path == 0 && plan_needs_cluster(elem_bytes, V)))
        return launch_ce_rows_long(grad, elem_bytes, prm, stream);
    // Aligned: every row (base + i * ld elements) starts on 16 bytes and ends on a vector.
    const bool aligned = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ld * elem_bytes) % 16 == 0 &&
                         (V * elem_bytes) % 16 == 0 && (dx == x || dx == nullptr || !grad);
    // Aligned rows of one slice, forward: the kernel whose warps run independently
    // (measured 58.0 -> 56.3 us on the 4096 x 32000 bf16 batch); the fused sweep
    // stays on the CTA kernel below (95.0 against 104 us); the test hook's 3 forces it.
    static const bool threads_forced = std::getenv("FOAK_ROW_THREADS") != nullptr;
    if (aligned && warp_ok && (hook == 3 || !grad) && !threads_forced && ce_rows_warp_fits(elem_bytes, V))
        return launch_ce_rows_warp(grad, elem_bytes, prm, stream);
    if (elem_bytes == 2)
        return grad ? launch_vpt<2, true>(prm, pl, stream, aligned) : launch_vpt<2, false>(prm, pl, stream, aligned);
    return grad ? launch_vpt<4, true>(prm, pl, stream, aligned) : launch_vpt<4, false>(prm, pl, stream, aligned);
}

}  // namespace foak
