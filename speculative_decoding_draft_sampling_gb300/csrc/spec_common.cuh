// spec_common.cuh -- device helpers shared by the verification kernels:
// inline-PTX wrappers for mbarriers and 1-D TMA bulk copies (sm_90+ / sm_103a),
// bounded waits, order-preserving sort keys, warp and block reductions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace spec {

#ifndef SPEC_THREADS
#define SPEC_THREADS 384
#endif
#ifndef SPEC_CTAS_PER_SM
#define SPEC_CTAS_PER_SM 2
#endif
constexpr int kThreads = SPEC_THREADS;        // consumer threads of every engine CTA
constexpr int kCtasPerSm = SPEC_CTAS_PER_SM;  // engine CTAs resident per SM (register and smem budget)
constexpr int kWarps = kThreads / 32;         // consumer warps
constexpr int kProducer = kThreads;           // the producer lane (warp kWarps, lane 0)
constexpr int kCombiner0 = kThreads + 32;     // first thread of the combiner warp (warp kWarps + 1)
constexpr int kBlockThreads = kThreads + 64;  // consumers + producer warp + combiner warp

// Barrier among the consumer threads only (named barrier 1; the producer
// warp never takes part), with the memory ordering of __syncthreads().
__device__ __forceinline__ void csync() {
    asm volatile("bar.sync 1, %0;" :: "n"(kThreads) : "memory");
}
// the same, returning whether any consumer thread passed a non-zero value
__device__ __forceinline__ int csync_or(int p) {
    int r;
    asm volatile(
        "{\n\t.reg .pred a, b;\n\t"
        "setp.ne.s32 a, %1, 0;\n\t"
        "bar.red.or.pred b, 1, %2, a;\n\t"
        "selp.s32 %0, 1, 0, b;\n\t}"
        : "=r"(r) : "r"(p), "n"(kThreads) : "memory");
    return r;
}
constexpr uint32_t kWaitLimit = 1u << 22;     // queue-wait polls (with backoff): ~seconds, never forever
// an mbarrier wait gives up after 2 s (test builds may shorten it)
#ifndef SPEC_WAIT_LIMIT_NS
#define SPEC_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr unsigned long long kMbarLimitNs = SPEC_WAIT_LIMIT_NS;
constexpr uint32_t kMbarPollLimit = 1u << 26;                  // ... or after this many polls
constexpr float kInf = __builtin_huge_valf();

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
struct F32 {
    using T = float;
    static constexpr int kBytes = 4;
    static constexpr int kVec = 4;            // elements per 16-byte vector
    __device__ static __forceinline__ void unpack(const uint4& w, float (&v)[4]) {
        v[0] = __uint_as_float(w.x); v[1] = __uint_as_float(w.y);
        v[2] = __uint_as_float(w.z); v[3] = __uint_as_float(w.w);
    }
    __device__ static __forceinline__ float load(const void* base, long long i) {
        return static_cast<const float*>(base)[i];
    }
};
struct BF16 {
    using T = __nv_bfloat16;
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
    __device__ static __forceinline__ void unpack(const uint4& w, float (&v)[8]) {
        v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xffff0000u);
        v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xffff0000u);
        v[4] = __uint_as_float(w.z << 16); v[5] = __uint_as_float(w.z & 0xffff0000u);
        v[6] = __uint_as_float(w.w << 16); v[7] = __uint_as_float(w.w & 0xffff0000u);
    }
    __device__ static __forceinline__ float load(const void* base, long long i) {
        uint32_t h = static_cast<const uint16_t*>(base)[i];
        return __uint_as_float(h << 16);
    }
};

// ---------------------------------------------------------------------------
// memory-model helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
// 128-bit record halves: each 64-bit half is single-copy atomic (a reader
// that needs both waits until neither reads zero)
__device__ __forceinline__ void ld_relaxed_v2(const unsigned long long* p, unsigned long long& a,
                                              unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_relaxed_v2(unsigned long long* p, unsigned long long a, unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
// release/acquire fence at GPU scope (orders this thread's, and by
// cumulativity the CTA's barrier-ordered, memory operations)
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void nanosleep_ns(uint32_t ns) {
    asm volatile("nanosleep.u32 %0;" :: "r"(ns));
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk copy (TMA), global -> shared
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// plain arrive (release at CTA scope)
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// copy `bytes` (multiple of 16, both addresses 16-byte aligned) and count the
// bytes on `bar`
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// one non-blocking test of the phase with the given parity
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// bounded wait for the phase with the given parity (2 s of wall time or
// kMbarPollLimit polls, whichever comes first); false when it gave up
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    unsigned long long t0 = 0;
    for (uint32_t it = 0; it < kMbarPollLimit; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        if (ok) return true;
        if ((it & 255u) == 255u) {
            const unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kMbarLimitNs) return false;
        }
    }
    return false;
}

// ---------------------------------------------------------------------------
// thread-block clusters: ranks, distributed shared memory, remote mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// the shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t mapa(uint32_t local_smem, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem), "r"(rank));
    return r;
}
// A load through a 32-bit shared-window address (data that reaches a
// function through a generic pointer would otherwise take the generic path).
__device__ __forceinline__ uint64_t lds_u64(uint32_t a) {
    uint64_t v;
    asm("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
// A read-only global load issued where it stands (the compiler may not sink
// it towards its first use), so that its latency overlaps the work between.
__device__ __forceinline__ uint32_t ldg_now_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_now_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
// Store 16 bytes into the shared memory of a CTA of the cluster (address
// from mapa) and count them on that CTA's mbarrier `bar` (complete_tx): the
// bytes are visible to a thread that observes the barrier's phase complete,
// with no fence on the storing side.  Both addresses in the same CTA; `a`
// 16-byte aligned.
__device__ __forceinline__ void st_async_v4(uint32_t a, const uint4& v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                 :: "r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar) : "memory");
}
// One arrival on a barrier of any CTA of the cluster that also expects
// `bytes` of st_async_v4 stores (from any thread of this CTA, before or after
// the arrival): the phase completes once every arrival is in and the bytes
// have landed.  Relaxed: it orders none of this thread's other accesses.
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}
// one non-blocking test of a phase completed by arrivals from other CTAs
// (acquire at cluster scope: their writes before the arrive are visible)
__device__ __forceinline__ bool mbar_test_cluster(const uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "r"(parity) : "memory");
    return ok != 0;
}
// every thread of every CTA of the cluster
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// keys: order-preserving uint32 of a float (-0 folded onto +0), and a 64-bit
// composite key ordering by value descending then index ascending (larger
// key = earlier in that order)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t fkey(float v) {
    uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}
__device__ __forceinline__ uint64_t ckey(float v, int x) {
    return (static_cast<uint64_t>(fkey(v)) << 32) | static_cast<uint32_t>(0x7fffffff - x);
}
__device__ __forceinline__ float ckey_val(uint64_t k) { return fkey_inv(static_cast<uint32_t>(k >> 32)); }
__device__ __forceinline__ int ckey_idx(uint64_t k) { return 0x7fffffff - static_cast<int>(static_cast<uint32_t>(k)); }

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ uint32_t warp_or(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Reductions over the kThreads consumer threads; `red` is shared scratch of
// at least kWarps 8-byte slots.  Every consumer thread receives the result.
__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, uint64_t* red) {
    v = warp_max_u64(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    csync();
    if (l == 0) red[w] = v;
    csync();
    uint64_t r = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) r = red[i] > r ? red[i] : r;
    return r;
}
__device__ __forceinline__ double block_sum_d(double v, double* red) {
    v = warp_sum_d(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    csync();
    if (l == 0) red[w] = v;
    csync();
    double r = 0.0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) r += red[i];
    return r;
}
__device__ __forceinline__ int block_sum_i(int v, int* red) {
    v = warp_sum_i(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    csync();
    if (l == 0) red[w] = v;
    csync();
    int r = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) r += red[i];
    return r;
}
__device__ __forceinline__ uint32_t block_or(uint32_t v, uint32_t* red) {
    v = warp_or(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    csync();
    if (l == 0) red[w] = v;
    csync();
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) r |= red[i];
    return r;
}
// warp-wide helpers (all 32 lanes)
__device__ __forceinline__ double warp_exscan_d(double v, double& total) {
    const int l = threadIdx.x & 31;
    double inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, inc, o);
        if (l >= o) inc += t;
    }
    total = __shfl_sync(0xffffffffu, inc, 31);
    return inc - v;
}
__device__ __forceinline__ int warp_exscan_i(int v, int& total) {
    const int l = threadIdx.x & 31;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (l >= o) inc += t;
    }
    total = __shfl_sync(0xffffffffu, inc, 31);
    return inc - v;
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) { return __reduce_max_sync(0xffffffffu, v); }
__device__ __forceinline__ uint32_t warp_min_u32(uint32_t v) { return __reduce_min_sync(0xffffffffu, v); }

// exclusive prefix sum (fp64) of one value per thread, in thread order; also
// returns the block total.
__device__ __forceinline__ double block_exscan_d(double v, double* red, double& total) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    double inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        double t = __shfl_up_sync(0xffffffffu, inc, o);
        if (l >= o) inc += t;
    }
    csync();
    if (l == 31) red[w] = inc;
    csync();
    double base = 0.0, tot = 0.0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
        if (i < w) base += red[i];
        tot += red[i];
    }
    total = tot;
    return base + inc - v;
}

// ---------------------------------------------------------------------------
// float-float ("double-single") sums: fp64 arithmetic is slow on this part,
// so sums that need more than fp32 keep a pair (hi, lo) with hi = fl(hi+lo),
// combined with the error-free two-sum (Knuth) -- about 48 significand bits
// with fp32 operations only.  Explicit _rn intrinsics keep the compiler from
// fusing or reordering the steps.
// ---------------------------------------------------------------------------
struct dfloat {
    float hi, lo;
};
__device__ __forceinline__ dfloat df_make(float x) { return {x, 0.f}; }
__device__ __forceinline__ dfloat df_add(dfloat a, dfloat b) {
    const float s = __fadd_rn(a.hi, b.hi);
    const float bb = __fsub_rn(s, a.hi);
    const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
    const float t = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    const float hi = __fadd_rn(s, t);
    return {hi, __fsub_rn(t, __fsub_rn(hi, s))};
}
__device__ __forceinline__ dfloat df_add(dfloat a, float b) { return df_add(a, df_make(b)); }
__device__ __forceinline__ dfloat df_neg(dfloat a) { return {-a.hi, -a.lo}; }
// x * y for fp32 x and a float-float y (error-free product of the hi parts)
__device__ __forceinline__ dfloat df_mul(float x, dfloat y) {
    const float p = __fmul_rn(x, y.hi);
    const float e = __fmaf_rn(x, y.hi, -p);
    const float t = __fmaf_rn(x, y.lo, e);
    const float hi = __fadd_rn(p, t);
    return {hi, __fsub_rn(t, __fsub_rn(hi, p))};
}
__device__ __forceinline__ bool df_gt(dfloat a, dfloat b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ double df_to_d(dfloat a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }
__device__ __forceinline__ dfloat df_from_d(double d) {
    const float hi = static_cast<float>(d);
    return {hi, static_cast<float>(d - static_cast<double>(hi))};
}
__device__ __forceinline__ dfloat warp_sum_df(dfloat v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        dfloat w;
        w.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        v = df_add(v, w);
    }
    return v;
}
// exclusive prefix (in lane order) and total
__device__ __forceinline__ dfloat warp_exscan_df(dfloat v, dfloat& total) {
    const int l = threadIdx.x & 31;
    dfloat inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        dfloat t;
        t.hi = __shfl_up_sync(0xffffffffu, inc.hi, o);
        t.lo = __shfl_up_sync(0xffffffffu, inc.lo, o);
        if (l >= o) inc = df_add(inc, t);
    }
    total.hi = __shfl_sync(0xffffffffu, inc.hi, 31);
    total.lo = __shfl_sync(0xffffffffu, inc.lo, 31);
    dfloat ex;
    ex.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
    ex.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
    if (l == 0) ex = df_make(0.f);
    return ex;
}
// consumers: sum over every consumer thread (red: kWarps float2 of shared scratch)
__device__ __forceinline__ dfloat block_sum_df(dfloat v, float2* red) {
    v = warp_sum_df(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    csync();
    if (l == 0) red[w] = make_float2(v.hi, v.lo);
    csync();
    dfloat r = df_make(0.f);
#pragma unroll
    for (int i = 0; i < kWarps; ++i) r = df_add(r, dfloat{red[i].x, red[i].y});
    return r;
}
// consumers: exclusive prefix in thread order, and the total
__device__ __forceinline__ dfloat block_exscan_df(dfloat v, float2* red, dfloat& total) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    dfloat wt;
    const dfloat ex = warp_exscan_df(v, wt);
    csync();
    if (l == 0) red[w] = make_float2(wt.hi, wt.lo);
    csync();
    dfloat base = df_make(0.f), tot = df_make(0.f);
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
        const dfloat x{red[i].x, red[i].y};
        if (i < w) base = df_add(base, x);
        tot = df_add(tot, x);
    }
    total = tot;
    return df_add(base, ex);
}

// max with NaN propagation (PTX max.NaN.f32): a NaN anywhere survives
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
template <int N>
__device__ __forceinline__ float vmax_nan(const float (&v)[N]) {
    float m = v[0];
#pragma unroll
    for (int j = 1; j < N; ++j) m = max_nan(m, v[j]);
    return m;
}

// fast 2^x on the special-function unit (PTX ex2.approx.ftz.f32)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace spec
