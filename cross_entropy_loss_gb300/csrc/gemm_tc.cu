// Persistent bf16 GEMM on the fifth-generation tensor cores (tcgen05) for the
// chunked linear + cross-entropy:  C (+)= A * B^T  with fp32 accumulation.
//
// Two kernels share the warp roles and the epilogue:
//   gemm_bf16_tc_kernel       one CTA per SM, output tiles of 128 x 256 (used when M
//                             has a single 128-row tile);
//   gemm_bf16_tc_pair_kernel  clusters of two CTAs whose tensor cores compute one
//                             256 x 256 tile together (tcgen05 cta_group::2): each
//                             CTA loads its own 128 rows of A and its own 128 rows of
//                             B (plain tiled TMA of its own tiles), the even CTA issues the
//                             M = 256 MMAs over both CTAs' shared memory, and each
//                             CTA's TMEM receives its 128 rows of the accumulator.
//                             Per CTA a 64-deep k-block is 32 KB instead of 48 KB, so
//                             the ring holds 6 stages and each SM reads a third less
//                             operand data from L2 per MMA.
// Warp roles:
//   warp 0     TMA producer: 2-D tiled loads (128-byte swizzle) of the A and B
//              k-blocks into a shared-memory ring;
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and
//              one thread issues tcgen05.mma per 16-deep slice, committing each
//              stage back to the producer(s) and each finished accumulator to the
//              epilogue(s);
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quarter of the accumulator,
//              then bf16 store (optionally with per-row softmax statistics of the
//              tile), fp32 store or fp32 reduce-add through the TMA engine.
// The accumulators are double-buffered, so a tile's epilogue overlaps the next
// tile's main loop.  Tiles are walked along the shorter tile dimension first (M
// fastest when there are fewer M tiles than N tiles, else N fastest), so the CTAs
// working at once share a few tiles of the operand with many tiles and every
// operand tile is fetched from HBM about once: for dW (250 x 16 tiles) an
// M-fastest walk re-read the 131 MB dZ operand once per N tile.  Either operand
// may be K-major (row-major [rows][K]) or MN-major (row-major [K][rows]); the
// shared-memory descriptors and the instruction descriptor's major bits say
// which.  All waits are bounded.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <type_traits>
#include <vector>

#include "foak_ce.h"
#include "gemm_tc.h"
#include "internal.h"
#include "tc.cuh"

namespace foak {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr uint32_t kABytes = kBM * kBK * 2;            // 16 KB: 128 rows of A
constexpr uint32_t kBBytes = kBN * kBK * 2;            // 32 KB: 256 rows of B
constexpr uint32_t kBHalfBytes = kBBytes / 2;          // a pair CTA's 128 rows of B
constexpr uint32_t kMNBlock = 64 * kBK * 2;            // one 64 (MN) x 64 (K) box: 8 KB
constexpr int kStages1 = 4;                            // single CTA: 48 KB stages
constexpr int kStages2 = 6;                            // pair CTA: 32 KB stages
constexpr uint32_t kStageBytes1 = kABytes + kBBytes;
constexpr uint32_t kStageBytes2 = kABytes + kBHalfBytes;
constexpr int kGemmThreads = 192;
constexpr uint32_t kTmemCols = 2 * kBN;
// fp32 outputs leave through shared memory: per epilogue warp two 32 x 32 fp32
// staging boxes (4 KB each, 128-byte swizzle) written back by TMA store or reduce-add.
constexpr uint32_t kStageOutBytes = 32 * 32 * 4;
constexpr uint32_t kOutStaging = 4 * 2 * kStageOutBytes;
constexpr size_t kGemmSmem1 = kStages1 * kStageBytes1 + kOutStaging + 1024;  // + alignment slack
constexpr size_t kGemmSmem2 = kStages2 * kStageBytes2 + kOutStaging + 1024;

struct GemmParams {
    CUtensorMap tmA;
    CUtensorMap tmB;
    CUtensorMap tmC;  // fp32 output (modes kGemmOutF32 / kGemmOutF32Acc)
    int M, N, K;
    int a_mn, b_mn;
    int mode;
    int units_m, tiles_n;  // output units: 128-row (single) or 256-row (pair) by 256 columns
    int n_fast;            // unit walk: N index fastest (else M)
    uint32_t idesc;
    void* out;
    int64_t ldo;
    int32_t* err;
    const int64_t* labels;  // statistics mode
    float2* stats;
    int stats_ld;
    float* zlab;
};
static_assert(kBN == kGemmTileN, "statistics tiles are the output tiles");

// Several independent products in one launch of the pair kernel: cluster c takes the
// (problem, unit) entries ent[start[c] .. start[c + 1]) in that order, a list the host
// balances by estimated cost (k-blocks plus the epilogue), longest units first.
constexpr int kGroupMax = 3;
constexpr int kGroupMaxClusters = 128;
constexpr int kGroupMaxUnits = 8192;
constexpr int kGroupUnitBits = 14;  // entry = (problem << 14) | unit
struct GemmGroup {
    GemmParams prob[kGroupMax];
    int nprob;
    GemmSideDz side;  // side.rows == 0: none
    uint16_t start[kGroupMaxClusters + 1];
    uint16_t ent[kGroupMaxUnits];
};

// Output units walked along the shorter dimension first.
__device__ __forceinline__ int unit_m(const GemmParams& p, int t) { return p.n_fast ? t / p.tiles_n : t % p.units_m; }
__device__ __forceinline__ int unit_n(const GemmParams& p, int t) { return p.n_fast ? t % p.tiles_n : t / p.units_m; }

// Epilogue of one accumulator for this warp: its 32 TMEM lanes are rows row_blk ..
// row_blk + 31 of C, 256 columns from n0 (tile column tn).  bf16 store (statistics
// mode: also the row's (max, sum exp) over the tile and its label's logit), or fp32
// store / reduce-add through two staging boxes and the TMA engine.
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t taddr, int row_blk, int n0, int tn,
                                              int lane, float* out_stage, uint32_t& out_it) {
    const int row = row_blk + lane;
    // statistics mode: this row's running (max, sum of exp(c - max)) over the tile's
    // columns, in natural-log units, and its label (its logit is kept when it is a column here)
    const bool stats = p.mode == kGemmOutBf16Stats && row < p.M;
    float st_m = kNegInf, st_s = 0.f;
    const int64_t ylab = stats ? __ldg(p.labels + row) : -1;
    // TMEM -> registers one 32-column chunk ahead: chunk c + 1 is loading while
    // chunk c is converted and stored (two register sets, loop unrolled)
    uint32_t ra[32], rb[32];
    tc_ld32(taddr, ra);
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c) {
        uint32_t(&r)[32] = (c & 1) ? rb : ra;
        uint32_t(&rn)[32] = (c & 1) ? ra : rb;
        tc_wait_ld(r);
        if (c + 1 < kBN / 32) tc_ld32(taddr + static_cast<uint32_t>((c + 1) * 32), rn);
        const int col0 = n0 + c * 32;
        if (col0 >= p.N) continue;
        const bool full_chunk = col0 + 32 <= p.N;
        if (p.mode == kGemmOutBf16 || p.mode == kGemmOutBf16Stats) {
            if (row >= p.M) continue;
            if (stats) {
                const int nv = min(32, p.N - col0);
                float cm = kNegInf;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nv) cm = fmaxf(cm, __uint_as_float(r[j]));
                const float mn = fmaxf(st_m, cm);
                const float mb = mn * kLog2e;
                float cs = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nv) cs += ex2(fmaf(__uint_as_float(r[j]), kLog2e, -mb));
                st_s = st_s * ex2(fmaf(st_m, kLog2e, -mb)) + cs;
                st_m = mn;
                if (ylab >= col0 && ylab < col0 + nv) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j == ylab) p.zlab[row] = __uint_as_float(r[j]);
                }
            }
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row) * p.ldo + col0;
            if (full_chunk) {
                uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                    w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                    w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                    w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                    o4[v] = w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (col0 + j < p.N) o[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
            }
        } else if (row_blk < p.M) {
            // stage the 32 x 32 box (row = lane) with the 128-byte swizzle, then one
            // TMA store or reduce-add writes it back; two boxes alternate per warp
            float* sbuf = out_stage + (out_it & 1) * (kStageOutBytes / 4);
            ++out_it;
            if (lane == 0) bulk_wait_group_read_1();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4*>(sbuf + lane * 32 + ((j ^ (lane & 7)) * 4)) =
                    make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (p.mode == kGemmOutF32Acc) tma_reduce_add_2d(&p.tmC, sbuf, col0, row_blk);
                else tma_store_2d(&p.tmC, sbuf, col0, row_blk);
                bulk_commit_group();
            }
        }
    }
    if (stats) p.stats[static_cast<int64_t>(row) * p.stats_ld + tn] = make_float2(st_m, st_s);
}

// Shared-memory descriptors of one 16-deep slice kk of a stage: K-major operands
// advance 32 bytes inside the 128-byte swizzle row, MN-major ones 16 K-rows of 128 bytes.
__device__ __forceinline__ uint64_t slice_desc(uint32_t base, int mn_major, int kk) {
    return mn_major ? smem_desc_sw128(base + kk * 2048, kMNBlock, 1024) : smem_desc_sw128(base + kk * 32, 16, 1024);
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_bf16_tc_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kStages1], empty[kStages1], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit0 = static_cast<int>(blockIdx.x);
    const int unit_step = static_cast<int>(gridDim.x);
    if (tid == 0) {
        for (int s = 0; s < kStages1; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        fence_mbar_init();
        abort_sh = 0;
        prefetch_tensormap(&p.tmA);
        prefetch_tensormap(&p.tmB);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // barriers and TMEM set up; operands and outputs are touched only after the previous
    // kernel in the stream has completed (programmatic dependent launch).  Dependents are
    // not let in early: small kernels waiting on SMs beside the MMA warps slowed the
    // chunked call by 1%.
    griddep_wait();
    const uint32_t tbase = tmem_base_sh;
    const int num_units = p.units_m * p.tiles_n;
    const int nk = (p.K + kBK - 1) / kBK;

    auto give_up = [&]() {
        abort_sh = 1;
        if (p.err) atomicOr(p.err, FOAK_ERRBIT_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int t = unit0; t < num_units && !abort_sh; t += unit_step) {
                const int m0 = unit_m(p, t) * kBM, n0 = unit_n(p, t) * kBN;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u)) { give_up(); break; }
                    if (abort_sh) break;
                    unsigned char* sA = smem + static_cast<size_t>(stage) * kStageBytes1;
                    unsigned char* sB = sA + kABytes;
                    mbar_arrive_expect_tx(&full[stage], kStageBytes1);
                    const int k0 = kb * kBK;
                    if (!p.a_mn) {
                        tma_load_2d(sA, &p.tmA, k0, m0, &full[stage]);
                    } else {
                        tma_load_2d(sA, &p.tmA, m0, k0, &full[stage]);
                        tma_load_2d(sA + kMNBlock, &p.tmA, m0 + 64, k0, &full[stage]);
                    }
                    if (!p.b_mn) {
                        tma_load_2d(sB, &p.tmB, k0, n0, &full[stage]);
                    } else {
#pragma unroll
                        for (int j = 0; j < kBN / 64; ++j) tma_load_2d(sB + j * kMNBlock, &p.tmB, n0 + 64 * j, k0, &full[stage]);
                    }
                    if (++stage == kStages1) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int t = unit0; t < num_units && !abort_sh; t += unit_step) {
                if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u)) { give_up(); break; }
                tc_fence_after();
                const uint32_t d_tmem = tbase + static_cast<uint32_t>(acc * kBN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase)) { give_up(); break; }
                    tc_fence_after();
                    const uint32_t sA = smem_u32(smem + static_cast<size_t>(stage) * kStageBytes1);
                    const uint32_t sB = sA + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma_bf16(d_tmem, slice_desc(sA, p.a_mn, kk), slice_desc(sB, p.b_mn, kk), p.idesc,
                                    (kb | kk) != 0 ? 1u : 0u);
                    tc_commit(&empty[stage]);
                    if (++stage == kStages1) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit(&acc_full[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else {
        // epilogue warps 2..5: TMEM lane quarter = warp % 4
        const int q = warp & 3;
        float* out_stage = reinterpret_cast<float*>(smem + kStages1 * kStageBytes1) + q * 2 * (kStageOutBytes / 4);
        uint32_t out_it = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = unit0; t < num_units; t += unit_step) {
            const bool ok = !abort_sh && mbar_wait_bounded(&acc_full[acc], acc_phase);
            if (!ok) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            const int tn = unit_n(p, t);
            const uint32_t taddr = tbase + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
            epilogue_tile(p, taddr, unit_m(p, t) * kBM + q * 32, tn * kBN, tn, lane, out_stage, out_it);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait_group_0();  // staged fp32 boxes fully written
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// CTA pairs (clusters of 2) on 256 x 256 output units.  CTA rank r holds rows
// m0 + 128r .. m0 + 128r + 127 of the unit's A and rows n0 + 128r .. of its B; the
// even CTA's full barriers count both CTAs' bytes (the odd CTA's copies complete on
// them), its MMA thread commits each stage to both CTAs' empty barriers and each
// accumulator to both CTAs' acc_full barriers (one commit per barrier), and
// both CTAs' epilogue warps arrive on the even CTA's acc_empty barriers.
// The side job of a grouped launch for one epilogue warp (gw of nw): work items are
// (row, 256-vector segment); lane l takes vectors l, l + 32, ... of the segment, all
// eight loads first, then the gradient and 16-byte streaming stores.
__device__ __forceinline__ void side_dz(const GemmSideDz& s, int gw, int nw, int lane) {
    const int nvec = s.V / 8;
    const int nseg = (nvec + 255) / 256;
    const float Dd = s.denom_dev ? static_cast<float>(__ldg(s.denom_dev)) : s.denom;
    const float scale = s.g / Dd;
    const int items = s.rows * nseg;
    for (int it = gw; it < items; it += nw) {
        const int r = it / nseg, sg = it - r * nseg;
        const int64_t y = __ldg(s.labels + r);
        const bool valid = y != s.ignore_index && y >= 0 && y < s.V;
        uint4* zr = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(s.z) + static_cast<int64_t>(r) * s.ldz);
        const int v0 = sg * 256;
        if (!valid) {
            if (sg == 0 && lane == 0 && y != s.ignore_index && s.err) atomicOr(s.err, FOAK_ERRBIT_LABEL_RANGE);
            const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int v = v0 + lane + 32 * i;
                if (v < nvec) st_global_cs_v4(zr + v, zero);
            }
            continue;
        }
        const float c = __ldg(s.lse + r) * kLog2e;
        const int yv = static_cast<int>(y >> 3), ye = static_cast<int>(y & 7);
        uint4 x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int v = v0 + lane + 32 * i;
            if (v < nvec) x[i] = ld_global_v4(zr + v);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int v = v0 + lane + 32 * i;
            if (v < nvec) {
                const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
                float d[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    d[2 * k] = ex2(fmaf(bf16_lo(w[k]), kLog2e, -c)) * scale;
                    d[2 * k + 1] = ex2(fmaf(bf16_hi(w[k]), kLog2e, -c)) * scale;
                }
                if (v == yv) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (e == ye) d[e] -= scale;
                }
                st_global_cs_v4(zr + v, make_uint4(pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3]),
                                                   pack_bf16x2(d[4], d[5]), pack_bf16x2(d[6], d[7])));
            }
        }
    }
}

// GROUPED: the kernel's argument is a GemmGroup and each cluster walks its entries;
// otherwise one GemmParams whose units the clusters take round-robin.
template <bool GROUPED>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_tc_pair_kernel(const __grid_constant__ typename std::conditional<GROUPED, GemmGroup, GemmParams>::type g) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kStages2], empty[kStages2], acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool lead = rank == 0;
    const int cl = static_cast<int>(blockIdx.x >> 1);
    const int ncl = static_cast<int>(gridDim.x >> 1);
    // this cluster's units: how many, and the i-th one's problem and unit index
    int n_my;
    if constexpr (GROUPED) {
        n_my = g.start[cl + 1] - g.start[cl];
    } else {
        const int units = g.units_m * g.tiles_n;
        n_my = cl < units ? (units - 1 - cl) / ncl + 1 : 0;
    }
    auto unit_at = [&](int i, int& t) -> const GemmParams& {
        if constexpr (GROUPED) {
            const unsigned e = g.ent[g.start[cl] + i];
            t = static_cast<int>(e & ((1u << kGroupUnitBits) - 1u));
            return g.prob[e >> kGroupUnitBits];
        } else {
            t = cl + i * ncl;
            return g;
        }
    };
    int32_t* err_word;
    if constexpr (GROUPED) err_word = g.prob[0].err;
    else err_word = g.err;
    if (tid == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 8);  // the four epilogue warps of each CTA
        }
        fence_mbar_init();
        abort_sh = 0;
        if constexpr (GROUPED) {
            for (int q = 0; q < g.nprob; ++q) {
                prefetch_tensormap(&g.prob[q].tmA);
                prefetch_tensormap(&g.prob[q].tmB);
            }
        } else {
            prefetch_tensormap(&g.tmA);
            prefetch_tensormap(&g.tmB);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(&tmem_base_sh, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any copy, commit or remote arrive
    tc_fence_after();
    // barriers and TMEM set up; operands and outputs are touched only after the previous
    // kernel in the stream has completed (programmatic dependent launch).  Dependents are
    // not let in early: small kernels waiting on SMs beside the MMA warps slowed the
    // chunked call by 1%.
    griddep_wait();
    const uint32_t tbase = tmem_base_sh;

    auto give_up = [&]() {
        abort_sh = 1;
        if (err_word) atomicOr(err_word, FOAK_ERRBIT_TIMEOUT);
    };

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int i = 0; i < n_my && !abort_sh; ++i) {
                int t;
                const GemmParams& p = unit_at(i, t);
                const int nk = (p.K + kBK - 1) / kBK;
                const int m0 = unit_m(p, t) * (2 * kBM) + static_cast<int>(rank) * kBM;
                const int nb0 = unit_n(p, t) * kBN + static_cast<int>(rank) * (kBN / 2);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u)) { give_up(); break; }
                    if (abort_sh) break;
                    unsigned char* sA = smem + static_cast<size_t>(stage) * kStageBytes2;
                    unsigned char* sB = sA + kABytes;
                    if (lead) mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes2);
                    const uint32_t bar = mapa_u32(&full[stage], 0);
                    const int k0 = kb * kBK;
                    if (!p.a_mn) {
                        tma_load_2d_pair(sA, &p.tmA, k0, m0, bar);
                    } else {
                        tma_load_2d_pair(sA, &p.tmA, m0, k0, bar);
                        tma_load_2d_pair(sA + kMNBlock, &p.tmA, m0 + 64, k0, bar);
                    }
                    if (!p.b_mn) {
                        tma_load_2d_pair(sB, &p.tmB, k0, nb0, bar);
                    } else {
                        tma_load_2d_pair(sB, &p.tmB, nb0, k0, bar);
                        tma_load_2d_pair(sB + kMNBlock, &p.tmB, nb0 + 64, k0, bar);
                    }
                    if (++stage == kStages2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && lead) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int i = 0; i < n_my && !abort_sh; ++i) {
                int t;
                const GemmParams& p = unit_at(i, t);
                const int nk = (p.K + kBK - 1) / kBK;
                if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u)) { give_up(); break; }
                tc_fence_after();
                const uint32_t d_tmem = tbase + static_cast<uint32_t>(acc * kBN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait_bounded(&full[stage], phase)) { give_up(); break; }
                    tc_fence_after();
                    const uint32_t sA = smem_u32(smem + static_cast<size_t>(stage) * kStageBytes2);
                    const uint32_t sB = sA + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma_bf16_pair(d_tmem, slice_desc(sA, p.a_mn, kk), slice_desc(sB, p.b_mn, kk), p.idesc,
                                         (kb | kk) != 0 ? 1u : 0u);
                    tc_commit_pair(smem_u32(&empty[stage]));
                    tc_commit_pair(mapa_u32(&empty[stage], 1));
                    if (++stage == kStages2) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit_pair(smem_u32(&acc_full[acc]));
                tc_commit_pair(mapa_u32(&acc_full[acc], 1));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else {
        // epilogue warps 2..5 of each CTA: TMEM lane quarter = warp % 4 of this CTA's 128 rows
        const int q = warp & 3;
        float* out_stage = reinterpret_cast<float*>(smem + kStages2 * kStageBytes2) + q * 2 * (kStageOutBytes / 4);
        uint32_t out_it = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t lead_acc_empty0 = mapa_u32(&acc_empty[0], 0);
        const uint32_t lead_acc_empty1 = mapa_u32(&acc_empty[1], 0);
        if constexpr (GROUPED) {
            // idle until the first accumulator is ready: the side job first
            if (g.side.rows > 0) side_dz(g.side, static_cast<int>(blockIdx.x) * 4 + q, static_cast<int>(gridDim.x) * 4, lane);
        }
        for (int i = 0; i < n_my; ++i) {
            int t;
            const GemmParams& p = unit_at(i, t);
            const bool ok = !abort_sh && mbar_wait_bounded(&acc_full[acc], acc_phase);
            if (!ok) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            const int tn = unit_n(p, t);
            const uint32_t taddr = tbase + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
            epilogue_tile(p, taddr, unit_m(p, t) * (2 * kBM) + static_cast<int>(rank) * kBM + q * 32, tn * kBN, tn,
                          lane, out_stage, out_it);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc == 0 ? lead_acc_empty0 : lead_acc_empty1);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait_group_0();  // staged fp32 boxes fully written
    tc_fence_before();
    __syncthreads();
    // no CTA frees its TMEM or leaves while the pair's MMAs, copies or arrivals may still reach it
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tbase, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// Row-major bf16 [outer][inner] with row stride ld (elements), boxes of 64 inner x
// box_outer, 128-byte swizzle (the layout the descriptors above expect).
bool encode_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, int64_t ld, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {64, box_outer};
    cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major fp32 [rows][cols] output with row stride ld: 32 x 32 boxes, 128-byte
// swizzle (the staging layout of the epilogue).
bool encode_f32_out(CUtensorMap* m, void* ptr, uint64_t cols, uint64_t rows, int64_t ld) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

std::mutex g_gemm_mu;
bool g_gemm_attr[64] = {false};

}  // namespace

namespace {

// Kernel parameters of one product; pair = CTA pairs on 256-row units (M has at least two
// 128-row tiles).  False when a tensor map cannot be encoded or the description is invalid.
bool make_params(const GemmDesc& d, GemmParams& p, bool& pair) {
    p = GemmParams{};
    const int tiles_m = (d.M + kBM - 1) / kBM;
    pair = tiles_m >= 2;
    // K-major [rows][K]: inner K, boxes of 64 x (the CTA's rows); MN-major [K][rows]: inner rows, 64 x 64 boxes.
    bool ok = d.a_mn_major ? encode_bf16(&p.tmA, d.a, static_cast<uint64_t>(d.M), static_cast<uint64_t>(d.K), d.lda, 64)
                           : encode_bf16(&p.tmA, d.a, static_cast<uint64_t>(d.K), static_cast<uint64_t>(d.M), d.lda, kBM);
    ok = ok && (d.b_mn_major
                    ? encode_bf16(&p.tmB, d.b, static_cast<uint64_t>(d.N), static_cast<uint64_t>(d.K), d.ldb, 64)
                    : encode_bf16(&p.tmB, d.b, static_cast<uint64_t>(d.K), static_cast<uint64_t>(d.N), d.ldb,
                                  pair ? kBN / 2 : kBN));
    if (ok && (d.mode == kGemmOutF32 || d.mode == kGemmOutF32Acc))
        ok = encode_f32_out(&p.tmC, d.out, static_cast<uint64_t>(d.N), static_cast<uint64_t>(d.M), d.ldo);
    if (!ok) return false;
    p.M = d.M;
    p.N = d.N;
    p.K = d.K;
    p.a_mn = d.a_mn_major ? 1 : 0;
    p.b_mn = d.b_mn_major ? 1 : 0;
    p.mode = d.mode;
    p.units_m = pair ? (tiles_m + 1) / 2 : tiles_m;
    p.tiles_n = (d.N + kBN - 1) / kBN;
    p.n_fast = p.units_m > p.tiles_n ? 1 : 0;
    p.idesc = idesc_bf16_f32(pair ? 2 * kBM : kBM, kBN, p.a_mn, p.b_mn);
    p.out = d.out;
    p.ldo = d.ldo;
    p.err = d.err;
    p.labels = d.labels;
    p.stats = d.stats;
    p.stats_ld = d.stats_ld;
    p.zlab = d.zlab;
    return !(d.mode == kGemmOutBf16Stats && (!d.labels || !d.stats || !d.zlab || d.stats_ld < p.tiles_n));
}

int g_max_pairs[64] = {0};

// Kernel attributes once per device, and the number of CTA pairs resident at once.
cudaError_t gemm_setup(int* max_pairs) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_gemm_mu);
    if (!g_gemm_attr[dev]) {
        e = cudaFuncSetAttribute(gemm_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemmSmem1));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_bf16_tc_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kGemmSmem2));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_bf16_tc_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kGemmSmem2));
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kGemmThreads, 1, 1);
        cfg.dynamicSmemBytes = kGemmSmem2;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, gemm_bf16_tc_pair_kernel<false>, &cfg);
        if (e != cudaSuccess) return e;
        g_max_pairs[dev] = std::max(1, n);
        g_gemm_attr[dev] = true;
    }
    *max_pairs = g_max_pairs[dev];
    return cudaSuccess;
}

template <typename Arg>
cudaError_t launch_pair(const Arg& arg, int clusters, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent: barrier and TMEM set-up overlap the previous kernel's end
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kGemmSmem2;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if constexpr (std::is_same<Arg, GemmGroup>::value)
        return cudaLaunchKernelEx(&cfg, gemm_bf16_tc_pair_kernel<true>, arg);
    else
        return cudaLaunchKernelEx(&cfg, gemm_bf16_tc_pair_kernel<false>, arg);
}

// Estimated cost of one unit in k-blocks: its main loop plus about 8 k-blocks of
// epilogue not hidden behind the next unit (from the measured per-unit times of the
// chunked products: 500 k-blocks 195 us, 64 k-blocks + statistics 28 us, 32 k-blocks +
// fp32 reduce-add 15 us on one pair).
int unit_cost(const GemmParams& p) { return (p.K + kBK - 1) / kBK + 8; }

struct Schedule {
    int clusters;
    std::vector<uint16_t> start, ent;
};

// Longest units first, each to the cluster with the least estimated work so far (ties:
// the lowest cluster); units of one problem keep their walk order, so clusters working
// at the same time share operand tiles as in a single product.
Schedule build_schedule(const GemmParams* ps, int n, int max_pairs) {
    struct U {
        int cost, prob, t;
    };
    std::vector<U> us;
    for (int q = 0; q < n; ++q)
        for (int t = 0; t < ps[q].units_m * ps[q].tiles_n; ++t) us.push_back({unit_cost(ps[q]), q, t});
    std::stable_sort(us.begin(), us.end(), [](const U& a, const U& b) { return a.cost > b.cost; });
    Schedule s;
    s.clusters = std::max(1, std::min(std::min(max_pairs, kGroupMaxClusters), static_cast<int>(us.size())));
    std::vector<int64_t> load(static_cast<size_t>(s.clusters), 0);
    std::vector<std::vector<uint16_t>> lists(static_cast<size_t>(s.clusters));
    for (const U& u : us) {
        int best = 0;
        for (int c = 1; c < s.clusters; ++c)
            if (load[static_cast<size_t>(c)] < load[static_cast<size_t>(best)]) best = c;
        load[static_cast<size_t>(best)] += u.cost;
        lists[static_cast<size_t>(best)].push_back(static_cast<uint16_t>((u.prob << kGroupUnitBits) | u.t));
    }
    s.start.push_back(0);
    for (const auto& l : lists) {
        s.ent.insert(s.ent.end(), l.begin(), l.end());
        s.start.push_back(static_cast<uint16_t>(s.ent.size()));
    }
    return s;
}

std::mutex g_sched_mu;
std::map<std::vector<int>, Schedule> g_sched;  // by (pairs, per problem: K, mode, units_m, tiles_n)

}  // namespace

cudaError_t launch_gemm_bf16(const GemmDesc& d, cudaStream_t stream) {
    if (d.M <= 0 || d.N <= 0 || d.K <= 0) return cudaSuccess;
    GemmParams p;
    bool pair = false;
    if (!make_params(d, p, pair)) return cudaErrorInvalidValue;
    int max_pairs = 0;
    cudaError_t e = gemm_setup(&max_pairs);
    if (e != cudaSuccess) return e;
    const int units = p.units_m * p.tiles_n;
    if (!pair) {
        const int grid = std::min(units, device_sm_count());
        return launch_dependent(gemm_bf16_tc_kernel, dim3(grid), dim3(kGemmThreads), kGemmSmem1, stream, p);
    }
    return launch_pair(p, std::min(units, max_pairs), stream);
}

int gemm_group_schedule(const int64_t* mnk, int n, int pairs, int32_t* start, int32_t* ent, int ent_cap) {
    if (n < 1 || n > kGroupMax || pairs < 1 || !mnk || !start || !ent) return -1;
    GemmParams ps[kGroupMax] = {};
    int total = 0;
    for (int q = 0; q < n; ++q) {
        const int64_t M = mnk[3 * q], N = mnk[3 * q + 1], K = mnk[3 * q + 2];
        if (M <= kBM || N <= 0 || K <= 0 || M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff) return -1;
        ps[q].units_m = static_cast<int>((M + kBM - 1) / kBM + 1) / 2;
        ps[q].tiles_n = static_cast<int>((N + kBN - 1) / kBN);
        ps[q].K = static_cast<int>(K);
        total += ps[q].units_m * ps[q].tiles_n;
    }
    if (total > ent_cap) return -1;
    const Schedule s = build_schedule(ps, n, pairs);
    for (size_t i = 0; i < s.start.size(); ++i) start[i] = s.start[i];
    for (size_t i = 0; i < s.ent.size(); ++i) ent[i] = s.ent[i];
    return s.clusters;
}

bool gemm_group_fits(const GemmDesc* d, int n) {
    int total = 0, live = 0;
    for (int i = 0; i < n; ++i) {
        if (d[i].M <= 0 || d[i].N <= 0 || d[i].K <= 0) continue;
        const int tiles_m = (d[i].M + kBM - 1) / kBM;
        if (tiles_m < 2) return false;
        const int u = (tiles_m + 1) / 2 * ((d[i].N + kBN - 1) / kBN);
        if (u >= (1 << kGroupUnitBits)) return false;
        total += u;
        ++live;
    }
    return live <= kGroupMax && total <= kGroupMaxUnits;
}

cudaError_t launch_gemm_bf16_group(const GemmDesc* d, int n, cudaStream_t stream, const GemmSideDz* side) {
    // the non-empty products
    const GemmDesc* live[kGroupMax];
    int nl = 0;
    for (int i = 0; i < n; ++i) {
        if (d[i].M <= 0 || d[i].N <= 0 || d[i].K <= 0) continue;
        if (nl == kGroupMax) return cudaErrorInvalidValue;
        live[nl++] = &d[i];
    }
    if (nl == 0) return cudaSuccess;
    // the grouped kernel arguments (about 18 KB: kept off the stack of the caller's thread)
    thread_local GemmGroup grp;
    int total = 0;
    bool all_pair = true, small = true;
    for (int q = 0; q < nl; ++q) {
        bool pair = false;
        if (!make_params(*live[q], grp.prob[q], pair)) return cudaErrorInvalidValue;
        const int u = grp.prob[q].units_m * grp.prob[q].tiles_n;
        all_pair = all_pair && pair;
        small = small && u < (1 << kGroupUnitBits);
        total += u;
    }
    const bool has_side = side && side->rows > 0;
    if (has_side && (!all_pair || !small || total > kGroupMaxUnits || side->V % 8 != 0 || side->ldz % 8 != 0 ||
                     reinterpret_cast<uintptr_t>(side->z) % 16 != 0))
        return cudaErrorInvalidValue;  // the caller checks gemm_group_fits and runs the job by itself otherwise
    // one product, a product of single-CTA tiles, or too many units: separate launches, in order
    if ((nl == 1 && !has_side) || !all_pair || !small || total > kGroupMaxUnits) {
        for (int q = 0; q < nl; ++q) {
            const cudaError_t e = launch_gemm_bf16(*live[q], stream);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    int max_pairs = 0;
    cudaError_t e = gemm_setup(&max_pairs);
    if (e != cudaSuccess) return e;
    std::vector<int> key = {max_pairs, nl};
    for (int q = 0; q < nl; ++q) {
        const GemmParams& p = grp.prob[q];
        key.insert(key.end(), {p.K, p.mode, p.units_m, p.tiles_n});
    }
    const Schedule* s = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_sched_mu);
        auto it = g_sched.find(key);
        if (it == g_sched.end()) it = g_sched.emplace(key, build_schedule(grp.prob, nl, max_pairs)).first;
        s = &it->second;
    }
    grp.nprob = nl;
    grp.side = has_side ? *side : GemmSideDz{};
    std::copy(s->start.begin(), s->start.end(), grp.start);
    std::copy(s->ent.begin(), s->ent.end(), grp.ent);
    return launch_pair(grp, s->clusters, stream);
}

}  // namespace foak
