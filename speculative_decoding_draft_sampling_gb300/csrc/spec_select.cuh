// spec_select.cuh -- per-slice pass functors for stream_row():
//   ArgmaxFn   max value with the lowest index (greedy, tree walk)
//   SumExpFn   max and sum of 2^((l - m) c), c = log2(e)/T (untruncated p)
//   TopkFn     all elements that can belong to the slice's top-k, found in one
//              pass with a running lower bound, then an exact selection
//   ResidFn    sum of [p - q]_+ and of the p weights (two streams)
// and the exact rank-based selections they and the combines use.
#pragma once

#include "spec_engine.cuh"

namespace spec {

// ---------------------------------------------------------------------------
// warp bitonic sort, descending, one 64-bit key per lane
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool lower = (lane & j) == 0;
            const bool first_half = (lane & k) == 0;
            const bool take_max = (lower == first_half);
            v = take_max ? (o > v ? o : v) : (o < v ? o : v);
        }
    }
    return v;
}

// ---------------------------------------------------------------------------
// exact selection from a shared-memory key array (keys unique)
// ---------------------------------------------------------------------------
// Ranks live in registers: kPer keys per thread (n <= kPer * kThreads).
// Keeps min(n, k) keys, or -- with `ties` -- every key whose value (high 32
// bits) is >= that of the k-th; writes them back sorted descending to
// cand[0 .. keep).  Returns keep; `kth` = key of rank k-1 (0 when n < k).
template <int kPer>
__device__ int select_inplace(uint64_t* cand, int n, int k, bool ties, uint64_t& kth,
                              uint64_t* sh64, int* ired) {
    uint64_t key[kPer];
    int rank[kPer];
    if (threadIdx.x == 0) sh64[0] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int i = threadIdx.x + j * kThreads;
        rank[j] = 0x7fffffff;
        key[j] = 0;
        if (i < n) {
            key[j] = cand[i];
            int r = 0;
            for (int t = 0; t < n; ++t) r += (cand[t] > key[j]);
            rank[j] = r;
            if (r == k - 1) sh64[0] = key[j];
        }
    }
    __syncthreads();
    kth = sh64[0];
    int keep;
    if (n < k) {
        keep = n;
    } else if (!ties) {
        keep = k;
    } else {
        const uint32_t th = static_cast<uint32_t>(kth >> 32);
        int c = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j)
            if (rank[j] != 0x7fffffff && static_cast<uint32_t>(key[j] >> 32) >= th) ++c;
        keep = block_sum_i(c, ired);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPer; ++j)
        if (rank[j] < keep) cand[rank[j]] = key[j];
    __syncthreads();
    return keep;
}

// Same selection with ranks in shared memory (large n, e.g. a combine over
// many slices): src[0..n) -> dst[0..keep) sorted descending.  keep is capped
// at dst_cap; *overflow set when the ties rule wanted more.
__device__ inline int select_to(const uint64_t* src, int n, int k, bool ties, int* rank,
                         uint64_t* dst, int dst_cap, uint64_t& kth, bool& overflow,
                         uint64_t* sh64, int* ired) {
    if (threadIdx.x == 0) sh64[0] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint64_t me = src[i];
        int r = 0;
        for (int t = 0; t < n; ++t) r += (src[t] > me);
        rank[i] = r;
        if (r == k - 1) sh64[0] = me;
    }
    __syncthreads();
    kth = sh64[0];
    int keep;
    if (n < k) {
        keep = n;
    } else if (!ties) {
        keep = k;
    } else {
        const uint32_t th = static_cast<uint32_t>(kth >> 32);
        int c = 0;
        for (int i = threadIdx.x; i < n; i += kThreads) c += (static_cast<uint32_t>(src[i] >> 32) >= th);
        keep = block_sum_i(c, ired);
    }
    overflow = keep > dst_cap;
    if (overflow) keep = dst_cap;
    for (int i = threadIdx.x; i < n; i += kThreads)
        if (rank[i] < keep) dst[rank[i]] = src[i];
    __syncthreads();
    return keep;
}

// ---------------------------------------------------------------------------
// functors
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bad_value(float v) {
    return (v != v) || (v == kInf);
}

template <class E>
struct ArgmaxFn {
    static constexpr bool kPrepass = false;
    uint64_t best = 0;
    uint32_t bad = 0;
    __device__ __forceinline__ void pre_vec(bool, const float (&)[E::kVec], int) {}
    __device__ __forceinline__ void pre_scalar(bool, float, int) {}
    __device__ __forceinline__ void pre_end() {}
    __device__ __forceinline__ void vec(bool act, const float (&v)[E::kVec], int x) {
        if (!act) return;
#pragma unroll
        for (int j = 0; j < E::kVec; ++j) {
            bad |= bad_value(v[j]);
            const uint64_t k = ckey(v[j], x + j);
            best = k > best ? k : best;
        }
    }
    __device__ __forceinline__ void scalar(bool act, float v, int x) {
        if (!act) return;
        bad |= bad_value(v);
        const uint64_t k = ckey(v, x);
        best = k > best ? k : best;
    }
    __device__ __forceinline__ void round_end() {}
};

// max and sum of 2^((l - m_t) c) with a per-thread running max m_t
template <class E>
struct SumExpFn {
    static constexpr bool kPrepass = false;
    float c;
    float m = -kInf;
    float s = 0.f;
    uint32_t bad = 0;
    __device__ __forceinline__ void pre_vec(bool, const float (&)[E::kVec], int) {}
    __device__ __forceinline__ void pre_scalar(bool, float, int) {}
    __device__ __forceinline__ void pre_end() {}
    __device__ __forceinline__ void add(float lm, const float* v, int n) {
        if (lm > m) {
            s *= ex2((m - lm) * c);
            m = lm;
        }
        if (m == -kInf) return;   // every value so far is -inf
        for (int j = 0; j < n; ++j) s += ex2((v[j] - m) * c);
    }
    __device__ __forceinline__ void vec(bool act, const float (&v)[E::kVec], int) {
        if (!act) return;
        float lm = v[0];
        bad |= bad_value(v[0]);
#pragma unroll
        for (int j = 1; j < E::kVec; ++j) {
            lm = fmaxf(lm, v[j]);
            bad |= bad_value(v[j]);
        }
        if (lm > m) {
            s *= ex2((m - lm) * c);
            m = lm;
        }
        if (m == -kInf) return;
#pragma unroll
        for (int j = 0; j < E::kVec; ++j) s += ex2((v[j] - m) * c);
    }
    __device__ __forceinline__ void scalar(bool act, float v, int) {
        if (!act) return;
        bad |= bad_value(v);
        add(v, &v, 1);
    }
    __device__ __forceinline__ void round_end() {}
};

// Elements that can belong to the slice's top-k: a running lower bound
// `theta` on the slice's k-th largest key filters the stream; survivors go to
// a shared candidate buffer.  The bound starts as the k-th largest of the
// per-warp top-8 (or top-32) thread maxima of the first chunk -- each of those
// is a real element, so at least k elements reach it -- and is raised to the
// exact k-th largest candidate whenever the buffer fills up.
//   kTies = true : keep every element whose value equals the k-th value
//                  (the top-k set S of a target distribution)
//   kTies = false: keep exactly k by (value desc, index asc) (DDTree lists)
template <class E, bool kTies, int kCap>
struct TopkFn {
    static constexpr bool kPrepass = true;
    static constexpr int VEC = E::kVec;
    static constexpr int kPer = (kCap + kThreads - 1) / kThreads;
    uint64_t* cand;     // [kCap] shared
    int* cnt;           // shared counter
    int* oflow;         // shared flag
    uint64_t* pool;     // [kThreads] shared scratch
    uint64_t* sh64;
    int* ired;
    int k;
    uint64_t theta = 0;
    uint64_t tmax = 0;
    uint32_t bad = 0;

    __device__ __forceinline__ bool passes(uint64_t key) const {
        if (kTies) return static_cast<uint32_t>(key >> 32) >= static_cast<uint32_t>(theta >> 32);
        return key >= theta;
    }
    __device__ __forceinline__ void pre_vec(bool act, const float (&v)[VEC], int x) {
        if (!act) return;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const uint64_t key = ckey(v[j], x + j);
            tmax = key > tmax ? key : tmax;
        }
    }
    __device__ __forceinline__ void pre_scalar(bool act, float v, int x) {
        if (!act) return;
        const uint64_t key = ckey(v, x);
        tmax = key > tmax ? key : tmax;
    }
    __device__ void pre_end() {
        const int per = (k <= 64) ? 8 : 32;
        const int P = per * kWarps;
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        const uint64_t s = warp_sort_desc(tmax);
        if (lane < per) pool[w * per + lane] = s;
        if (threadIdx.x == 0) sh64[1] = 0;
        __syncthreads();
        if (k <= P && threadIdx.x < P) {
            const uint64_t me = pool[threadIdx.x];
            int r = 0;
            for (int t = 0; t < P; ++t) r += (pool[t] > me);
            if (r == k - 1 && me != 0) sh64[1] = me;
        }
        __syncthreads();
        theta = sh64[1];
        __syncthreads();
    }
    __device__ __forceinline__ void append(uint32_t m, const uint64_t* keys, int nk) {
        const int c = __popc(m);
        if (__ballot_sync(0xffffffffu, c != 0) == 0) return;
        const int lane = threadIdx.x & 31;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int base = 0;
        if (lane == 31) base = atomicAdd(cnt, incl);
        base = __shfl_sync(0xffffffffu, base, 31);
        int pos = base + incl - c;
        for (int j = 0; j < nk; ++j) {
            if ((m >> j) & 1u) {
                if (pos < kCap) cand[pos] = keys[j];
                else *oflow = 1;
                ++pos;
            }
        }
    }
    __device__ __forceinline__ void vec(bool act, const float (&v)[VEC], int x) {
        uint64_t keys[VEC];
        uint32_t m = 0;
        if (act) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                bad |= bad_value(v[j]);
                keys[j] = ckey(v[j], x + j);
                if (passes(keys[j])) m |= 1u << j;
            }
        }
        append(m, keys, VEC);
    }
    __device__ __forceinline__ void scalar(bool act, float v, int x) {
        uint64_t key[1] = {0};
        uint32_t m = 0;
        if (act) {
            bad |= bad_value(v);
            key[0] = ckey(v, x);
            if (passes(key[0])) m = 1;
        }
        append(m, key, 1);
    }
    // raise theta to the exact k-th candidate when the next round could overflow
    __device__ void round_end() {
        __syncthreads();
        const int n = *cnt;
        __syncthreads();   // every thread has read cnt before the next round appends
        if (n > kCap - kThreads * VEC && n <= kCap) {
            uint64_t kth;
            const int keep = select_inplace<kPer>(cand, n, k, kTies, kth, sh64, ired);
            if (threadIdx.x == 0) *cnt = keep;
            if (n >= k) theta = kth;
            __syncthreads();
        }
    }
    // final exact selection; returns keep (keys sorted descending in cand)
    __device__ int finish(uint64_t& kth) {
        __syncthreads();
        int n = *cnt;
        if (n > kCap) n = kCap;   // overflow already flagged
        return select_inplace<kPer>(cand, n, k, kTies, kth, sh64, ired);
    }
};

// [p - q]_+ and p weights over one row with known max m and normaliser Z
template <class E>
struct ResidFn {
    float m, c, invZ;
    float r = 0.f, pw = 0.f;
    __device__ __forceinline__ void vec2(bool act, const float (&lv)[E::kVec], const float (&qv)[E::kVec], int) {
        if (!act) return;
#pragma unroll
        for (int j = 0; j < E::kVec; ++j) {
            const float w = ex2((lv[j] - m) * c);
            const float d = w * invZ - qv[j];
            r += d > 0.f ? d : 0.f;
            pw += w;
        }
    }
    __device__ __forceinline__ void scalar2(bool act, float l, float q, int) {
        if (!act) return;
        const float w = ex2((l - m) * c);
        const float d = w * invZ - q;
        r += d > 0.f ? d : 0.f;
        pw += w;
    }
};

}  // namespace spec
