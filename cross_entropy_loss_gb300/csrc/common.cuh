// Device-side building blocks shared by the library's kernels: shared-memory
// barriers, bulk (TMA) copies, cluster barriers and distributed shared memory,
// written as inline PTX for sm_103a.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace foak {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_inff();

// Waits on shared-memory barriers give up after this long (a healthy wait is
// microseconds); the kernel then records FOAK_ERRBIT_TIMEOUT and winds down.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------ programmatic dependent launch
// A kernel launched with the programmatic-serialization attribute may start while the
// previous kernel in its stream is still running; griddep_wait() returns once that
// kernel has completed and its writes are visible, so no global memory may be touched
// before it.  Without the attribute it returns at once.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next such kernel in the stream be scheduled (it still waits in griddep_wait).
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// ------------------------------------------------ double-float sums of float terms
// A value carried as hi + lo in two floats.  Additions take Knuth's TwoSum (an exact
// error-free transform: s + e == a + b) and renormalise with Dekker's Fast2Sum, so a
// sum of float terms keeps about 48 significant bits on the FP32 pipe; the FP64 pipe
// of this part is narrow enough that a few dozen dependent float64 additions and a
// division at the end of a kernel cost microseconds.  Non-finite sums propagate as
// in plain float arithmetic.
struct DFloat {
    float hi, lo;
};

__device__ __forceinline__ DFloat df_add(DFloat x, float b) {
    const float s = __fadd_rn(x.hi, b);
    if (!isfinite(s)) return DFloat{s, 0.f};
    const float bp = __fsub_rn(s, x.hi);
    const float e = __fadd_rn(__fadd_rn(__fsub_rn(x.hi, __fsub_rn(s, bp)), __fsub_rn(b, bp)), x.lo);
    const float hi = __fadd_rn(s, e);
    return DFloat{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

__device__ __forceinline__ DFloat df_add(DFloat x, DFloat y) {
    DFloat r = df_add(x, y.hi);
    if (!isfinite(r.hi)) return r;
    const float hi = __fadd_rn(r.hi, y.lo);
    return DFloat{hi, __fadd_rn(r.lo, __fsub_rn(y.lo, __fsub_rn(hi, r.hi)))};
}

// (hi + lo) / d as a float: the quotient of hi, corrected by the remainder hi - q d,
// which an FMA gives exactly for a correctly rounded q, plus lo.
__device__ __forceinline__ float df_div(DFloat x, float d) {
    const float q = __fdiv_rn(x.hi, d);
    if (!isfinite(q)) return q;
    const float r = fmaf(-q, d, x.hi);
    return __fadd_rn(q, __fdiv_rn(__fadd_rn(r, x.lo), d));
}

// Sum of v[0, n) over a CTA of THREADS threads, in a fixed order: thread t adds
// v[t], v[t + THREADS], ... (eight loads in flight before their additions), then a
// shuffle tree per warp and the same tree over the warps' partials in warp 0.  `red` holds THREADS/32
// values; the result is valid in thread 0.  Loads bypass L1 (the terms were written
// by other CTAs of the same kernel).
template <int THREADS>
__device__ __forceinline__ DFloat block_sum_terms(const float* v, int64_t n, DFloat* red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    DFloat acc{0.f, 0.f};
    for (int64_t i0 = tid; i0 < n; i0 += 8 * THREADS) {
        float t[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t i = i0 + static_cast<int64_t>(k) * THREADS;
            t[k] = i < n ? __ldcg(v + i) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = df_add(acc, t[k]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const DFloat o{__shfl_down_sync(0xffffffffu, acc.hi, off), __shfl_down_sync(0xffffffffu, acc.lo, off)};
        acc = df_add(acc, o);
    }
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    // the warp partials by warp 0: the same shuffle tree over lanes 0 .. THREADS/32 - 1
    DFloat tot{0.f, 0.f};
    if (warp == 0) {
        static_assert(THREADS / 32 <= 32, "one partial per lane");
        tot = lane < THREADS / 32 ? red[lane] : DFloat{0.f, 0.f};
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const DFloat o{__shfl_down_sync(0xffffffffu, tot.hi, off), __shfl_down_sync(0xffffffffu, tot.lo, off)};
            tot = df_add(tot, o);
        }
    }
    return tot;
}

// Fetch-and-add with release and acquire semantics at GPU scope: earlier writes of this
// thread (and those it has seen) are visible before the add, and later reads see what
// the threads whose adds it follows had written.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test without the hardware's optional suspension of the waiting thread:
// for spin loops whose waits usually end within a few hundred cycles.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// when limit_ns (default kWaitLimitNs) elapsed first.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- bulk copies
// One-dimensional bulk copy global -> this CTA's shared memory, completing `bytes`
// transactions on `bar`.  Addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 eviction-priority policies for cache-hinted copies.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 eviction-priority hint for the lines it reads.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
    cluster_arrive_release();
    cluster_wait_acquire();
}

// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_u32(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    return remote;
}

// Asynchronous store of two floats into (possibly another CTA's) shared memory,
// completing 8 bytes of transaction on that CTA's mbarrier; no fence is implied.
__device__ __forceinline__ void st_async_f2(uint32_t remote_addr, float a, float b, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(remote_addr),
                 "f"(a), "f"(b), "r"(remote_bar)
                 : "memory");
}

// ---------------------------------------------------------------- math / memory
// 2^x on the special-function unit (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) on the special-function unit (PTX lg2.approx.ftz.f32).
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void st_global_cs_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_global_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// bf16 <-> f32 on packed words: element 0 is the low half.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- packed pairs
// Two floats in one 64-bit register pair, for the sm_100-family paired FP32
// instructions (fma/add/mul .f32x2), which do two lanes of work per issue.
typedef unsigned long long f32x2_t;

__device__ __forceinline__ f32x2_t f2_pack(float lo, float hi) {
    f32x2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(f32x2_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2_t f2_fma(f32x2_t a, f32x2_t b, f32x2_t c) {
    f32x2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2_t f2_add(f32x2_t a, f32x2_t b) {
    f32x2_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2_t f2_mul(f32x2_t a, f32x2_t b) {
    f32x2_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2_t f2_ex2(f32x2_t a) {
    float lo, hi;
    f2_unpack(a, lo, hi);
    return f2_pack(ex2(lo), ex2(hi));
}
// bf16 pair (low half = element 0) widened exactly to two floats.
__device__ __forceinline__ f32x2_t bf16x2_to_f2(uint32_t w) { return f2_pack(bf16_lo(w), bf16_hi(w)); }
// Two floats rounded to nearest-even bf16, packed with element 0 in the low half.
__device__ __forceinline__ uint32_t f2_to_bf16x2(f32x2_t v) {
    float lo, hi;
    f2_unpack(v, lo, hi);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}
// The same max in one warp-wide reduction instruction (redux.sync on f32, an
// sm_100-family feature) instead of five dependent shuffles: shorter latency,
// which pays off where the row's reduction chain is the critical path (the
// forward sweep, the two-pass kernel); all 32 lanes must be converged.
__device__ __forceinline__ float warp_max_redux(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Online (max, sum of exp(x - max)) pair merge, natural-log units.
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
    const float mn = fmaxf(m, m2);
    if (mn == kNegInf) return;  // both empty
    s = s * ex2((m - mn) * kLog2e) + s2 * ex2((m2 - mn) * kLog2e);
    m = mn;
}

__device__ __forceinline__ void warp_ms_reduce(float& m, float& s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        ms_merge(m, s, m2, s2);
    }
}

// Number of labels in [0, V) (valid) and of labels that are neither ignore_index
// nor in range (bad), counted by the whole CTA; every thread gets the totals.
// `scratch` holds 2 * (blockDim.x / 32) ints.
__device__ __forceinline__ void count_labels(const int64_t* __restrict__ labels, int64_t N, int64_t V,
                                             int64_t ignore_index, int* scratch, int& n_valid,
                                             int& n_bad) {
    int cv = 0, cb = 0;
    // eight independent loads in flight per thread, not one round trip per label
    for (int64_t i0 = threadIdx.x; i0 < N; i0 += 8 * static_cast<int64_t>(blockDim.x)) {
        int64_t y[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t i = i0 + static_cast<int64_t>(k) * blockDim.x;
            y[k] = i < N ? __ldg(labels + i) : ignore_index;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (y[k] != ignore_index) {
                if (y[k] >= 0 && y[k] < V) ++cv;
                else ++cb;
            }
        }
    }
    cv = __reduce_add_sync(0xffffffffu, cv);
    cb = __reduce_add_sync(0xffffffffu, cb);
    const int nw = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        scratch[threadIdx.x >> 5] = cv;
        scratch[nw + (threadIdx.x >> 5)] = cb;
    }
    __syncthreads();
    int tv = 0, tb = 0;
    for (int w = 0; w < nw; ++w) {
        tv += scratch[w];
        tb += scratch[nw + w];
    }
    n_valid = tv;
    n_bad = tb;
}

}  // namespace foak
