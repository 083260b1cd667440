// spec_select.cuh -- per-slice pass functors for stream_row():
//   ArgmaxFn    max value with the lowest index (greedy, tree walk)
//   SumExpFn    max and sum of 2^((l - m) c), c = log2(e)/T (untruncated p)
//   TopkHistFn  every element that can belong to the row's top-k, found in
//               one pass behind a certified (or hinted) value threshold
//   ResidFn     sum of [p - q]_+ and of the p weights (two streams)
// and the exact rank-based selection and histogram bounds the functors and
// the combines use.
#pragma once

#include "spec_engine.cuh"

namespace spec {

// value key of a composite key
__device__ __forceinline__ uint32_t hkey(uint64_t k) { return static_cast<uint32_t>(k >> 32); }

// Float threshold equivalent to a value-key threshold: for every non-NaN x,
// x >= key_to_thr(t)  <=>  fkey(x) >= t.
__device__ __forceinline__ float key_to_thr(uint32_t t) {
    if (t <= fkey(-kInf)) return -kInf;
    if (t >= fkey(kInf)) return kInf;
    return fkey_inv(t);
}

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
// number of keys in src[0..n) greater than `me`; src 16-byte aligned (two
// keys per shared load, every thread reading the same address)
__device__ __forceinline__ int count_greater(const uint64_t* src, int n, uint64_t me) {
    const ulonglong2* s2 = reinterpret_cast<const ulonglong2*>(src);
    int r = 0;
    const int n2 = n >> 1;
    for (int t = 0; t < n2; ++t) {
        const ulonglong2 p = s2[t];
        r += (p.x > me) + (p.y > me);
    }
    if (n & 1) r += src[n - 1] > me;
    return r;
}

// src[0..n) (16-byte aligned) -> dst[0..keep) sorted descending.  Keeps
// min(n, k) keys or -- with `ties` -- every key whose value (high 32 bits)
// reaches that of the k-th.  keep is capped at dst_cap; `overflow` is set
// when the ties rule wanted more.  `kth` = key of rank k-1 (0 when n < k).
// `rank` is shared scratch of n ints.
__device__ inline int select_to(const uint64_t* src, int n, int k, bool ties, int* rank,
                                uint64_t* dst, int dst_cap, uint64_t& kth, bool& overflow,
                                uint64_t* sh64, int* ired) {
    if (threadIdx.x == 0) sh64[0] = 0;
    csync();
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint64_t me = src[i];
        const int r = count_greater(src, n, me);
        rank[i] = r;
        if (r == k - 1) sh64[0] = me;
    }
    csync();
    kth = sh64[0];
    int keep;
    if (n < k) {
        keep = n;
    } else if (!ties) {
        keep = k;
    } else {
        const uint32_t th = hkey(kth);
        int c = 0;
        for (int i = threadIdx.x; i < n; i += kThreads) c += hkey(src[i]) >= th;
        keep = block_sum_i(c, ired);
    }
    overflow = keep > dst_cap;
    if (overflow) keep = dst_cap;
    for (int i = threadIdx.x; i < n; i += kThreads)
        if (rank[i] < keep) dst[rank[i]] = src[i];
    csync();
    return keep;
}

// ---------------------------------------------------------------------------
// certified histogram bound
// ---------------------------------------------------------------------------
// A lower bound B >= lo on the value key of the k-th largest key such that at
// least k keys have value key >= B: the lower edge of the highest bin of a
// 64-bin histogram over [lo, max] whose suffix count reaches k; a bottom bin
// holding the k-th is split again until it is one key wide.  `each(f)` calls
// f(value key) for every key this thread owns.  `certified` is set when at
// least k keys reach lo (then B is a bound for any superset of the keys).
// All threads; hist[64], scratch[kWarps + 1] shared.
template <class Each>
__device__ uint32_t hist_bound(Each each, int k, uint32_t lo, int* hist, uint32_t* scratch, bool& certified) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t mk = 0;
    each([&](uint32_t h) { mk = max(mk, h); });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    csync();
    if (lane == 0) scratch[w] = mk;
    csync();
    uint32_t top = scratch[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) top = max(top, scratch[i]);
    const uint32_t d = top > lo ? top - lo : 0u;
    const int bits = 32 - __clz(d);
    uint32_t sh = bits > 6 ? static_cast<uint32_t>(bits - 6) : 0u;
    uint32_t bound = lo;
    certified = false;
    for (int round = 0; round < 6; ++round) {
        for (int i = threadIdx.x; i < 64; i += kThreads) hist[i] = 0;
        csync();
        each([&](uint32_t h) {
            if (h >= lo) {
                const uint32_t bb = (h - lo) >> sh;
                atomicAdd(&hist[bb < 64 ? bb : 63], 1);
            }
        });
        csync();
        if (w == 0) {
            const int h0 = hist[2 * lane], h1 = hist[2 * lane + 1];
            int suf = h0 + h1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += t;
            }
            const int above = suf - h0 - h1;
            int best = -1;
            if (above + h1 >= k) best = 2 * lane + 1;
            else if (above + h1 + h0 >= k) best = 2 * lane;
            const uint32_t ql = __ballot_sync(0xffffffffu, best >= 0);
            const int bl = ql ? 31 - __clz(ql) : -1;
            const int bb = __shfl_sync(0xffffffffu, best, bl >= 0 ? bl : 0);
            if (lane == 0) scratch[kWarps] = static_cast<uint32_t>(bl >= 0 ? bb : -1);
        }
        csync();
        const int bb = static_cast<int>(scratch[kWarps]);
        csync();
        if (bb < 0) break;                 // fewer than k keys reach lo
        certified = true;
        if (bb > 0) {
            const uint64_t e = static_cast<uint64_t>(lo) + (static_cast<uint64_t>(bb) << sh);
            if (e <= 0xffffffffull) bound = static_cast<uint32_t>(e);
            break;
        }
        if (sh == 0) break;
        sh = sh >= 6 ? sh - 6 : 0u;
    }
    return bound;
}

// The largest composite key t >= lo64 with at least k keys >= t, when the
// k-th largest key has value key hkey(lo64) (so t differs from lo64 only in
// the index bits): bisection over the low 32 bits.  `each(f)` calls f(key)
// for every key this thread owns.  All threads; ired[kWarps] shared.
template <class Each>
__device__ uint64_t composite_bound(Each each, int k, uint64_t lo64, int* ired) {
    uint64_t lo = lo64, hi = lo64 | 0xffffffffull;
    for (int it = 0; it < 34 && lo < hi; ++it) {
        const uint64_t mid = lo + ((hi - lo + 1) >> 1);
        int c = 0;
        each([&](uint64_t key) { c += key >= mid; });
        c = block_sum_i(c, ired);
        if (c >= k) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// the same over a contiguous shared list
__device__ inline uint32_t hist_bound_list(const uint64_t* list, int n, int k, uint32_t lo, int* hist,
                                           uint32_t* scratch, bool& certified) {
    return hist_bound([&](auto f) { for (int i = threadIdx.x; i < n; i += kThreads) f(hkey(list[i])); },
                      k, lo, hist, scratch, certified);
}

// Keep the keys of list[0..n) with value key >= t, in place (order kept).
// All threads; returns the new count.  ired[kWarps + 1] shared.
__device__ inline int compact_list(uint64_t* list, int n, uint32_t t, int* ired) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int out = 0;
    for (int i0 = 0; i0 < n; i0 += kThreads) {
        const int i = i0 + threadIdx.x;
        uint64_t key = 0;
        bool p = false;
        if (i < n) { key = list[i]; p = hkey(key) >= t; }
        const uint32_t bal = __ballot_sync(0xffffffffu, p);
        if (lane == 0) ired[w] = __popc(bal);
        csync();
        int base = out;
        int tot = 0;
#pragma unroll
        for (int j = 0; j < kWarps; ++j) {
            const int c = ired[j];
            if (j < w) base += c;
            tot += c;
        }
        csync();   // every thread read its block before anyone writes
        if (p) list[base + __popc(bal & ((1u << lane) - 1u))] = key;
        out += tot;
        csync();
    }
    return out;
}

// ---------------------------------------------------------------------------
// functors
// ---------------------------------------------------------------------------
// a value that poisons a row: NaN or +inf (a running max_nan sees both)
__device__ __forceinline__ uint32_t bad_max(float vmx) { return !(vmx < kInf); }

// Max value, lowest index.  Per vector, a NaN-propagating max decides
// whether any element can beat the thread's best; only then are the elements
// examined.  Each thread sees its elements in increasing index order, so a
// strict > keeps the lowest index among equal values.
template <class E>
struct ArgmaxFn : FnHooks {
    float bv = -kInf;   // best value
    int bx = -1;        // its index
    float vmx = -kInf;  // running max with NaN propagation (bad-value test)
    __device__ __forceinline__ void vec(bool act, const float (&v)[E::kVec], int x) {
        if (!act) return;
        const float m4 = vmax_nan(v);
        vmx = max_nan(vmx, m4);
        if (!(m4 <= bv)) {
#pragma unroll
            for (int j = 0; j < E::kVec; ++j)
                if (v[j] > bv) { bv = v[j]; bx = x + j; }
        }
    }
    __device__ __forceinline__ void scalar(bool act, float v, int x) {
        if (!act) return;
        vmx = max_nan(vmx, v);
        if (v > bv) { bv = v; bx = x; }
    }
    // four rounds at once (vector r at x + r * kThreads * VEC): one test
    // decides whether any element can beat the thread's best; the rounds are
    // then examined in increasing index order, so the lowest index still wins
    static constexpr bool kVec4 = true;
    __device__ __forceinline__ void vec4(const float (&v)[4][E::kVec], int x) {
        const float m0 = vmax_nan(v[0]), m1 = vmax_nan(v[1]), m2 = vmax_nan(v[2]), m3 = vmax_nan(v[3]);
        const float mm = max_nan(max_nan(m0, m1), max_nan(m2, m3));
        vmx = max_nan(vmx, mm);
        if (!(mm <= bv)) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int j = 0; j < E::kVec; ++j)
                    if (v[r][j] > bv) { bv = v[r][j]; bx = x + r * kThreads * E::kVec + j; }
            }
        }
    }
    // composite key of the thread's best (0 when it saw no value above -inf)
    __device__ __forceinline__ uint64_t key() const { return bx >= 0 ? ckey(bv, bx) : 0ull; }
    __device__ __forceinline__ uint32_t bad_flag() const { return bad_max(vmx); }
};

// max and sum of 2^((l - m_t) c) with a per-thread running max m_t; with
// kMask only elements whose value key reaches `mask` are summed (the row's
// top-k set when its threshold is known; the running max is over every
// element, and the row maximum always belongs to the set)
template <class E, bool kMask = false>
struct SumExpFn : FnHooks {
    float c;
    float thr = -kInf;   // kMask: v >= thr  <=>  value key >= mask
    float m = -kInf;
    float s = 0.f;
    float vmx = -kInf;
    __device__ __forceinline__ void vec(bool act, const float (&v)[E::kVec], int) {
        if (!act) return;
        const float lm = vmax_nan(v);
        vmx = max_nan(vmx, lm);
        if (lm > m) {
            s *= ex2((m - lm) * c);
            m = lm;
        }
        if (m == -kInf) return;   // every value so far is -inf
#pragma unroll
        for (int j = 0; j < E::kVec; ++j) {
            if (kMask && !(v[j] >= thr)) continue;
            s += ex2((v[j] - m) * c);
        }
    }
    __device__ __forceinline__ void scalar(bool act, float v, int) {
        if (!act) return;
        vmx = max_nan(vmx, v);
        if (v > m) {
            s *= ex2((m - v) * c);
            m = v;
        }
        if (m == -kInf) return;
        if (kMask && !(v >= thr)) return;
        s += ex2((v - m) * c);
    }
    __device__ __forceinline__ uint32_t bad_flag() const { return bad_max(vmx); }
};

// Histogram of one 8-bit digit of the value keys (round r: bits 31-8r down
// to 24-8r) over the elements whose higher digits equal `prefix`: one round
// of an exact radix select of the row's k-th largest value.
template <class E>
struct RadixFn : FnHooks {
    int* bins;          // 256 shared counters, zeroed by the caller
    int round;
    uint32_t prefix;
    float vmx = -kInf;
    __device__ __forceinline__ void one(float v) {
        vmx = max_nan(vmx, v);
        const uint32_t k = fkey(v);
        const int sh = 24 - 8 * round;
        if (round == 0 || (k >> (sh + 8)) == prefix) atomicAdd(&bins[(k >> sh) & 255u], 1);
    }
    __device__ __forceinline__ void vec(bool act, const float (&v)[E::kVec], int) {
        if (!act) return;
#pragma unroll
        for (int j = 0; j < E::kVec; ++j) one(v[j]);
    }
    __device__ __forceinline__ void scalar(bool act, float v, int) {
        if (act) one(v);
    }
};

// Shared state of TopkHistFn: one candidate region per warp, so a warp
// appends with ballots and a register counter and never waits for the other
// warps.
struct TopkSmem {
    static constexpr int kRegion = 256;                 // keys per warp
    static constexpr int kSlots = 4;                    // per-thread keys within a chunk
    alignas(16) uint64_t cand[kWarps * kRegion];
    uint64_t slot[kSlots][kThreads];
    uint64_t pool[kThreads];
    uint64_t wthr[kWarps];
    float wmax[kWarps];
    int wn[kWarps];
    int hist[64];
    uint32_t scratch[kWarps + 2];
    uint64_t sh64[2];
    int ired[kWarps + 4];
    // the best certified value filter any warp found for the current unit:
    // (unit tag << 32) | value key; a stale tag is ignored.  Zero at kernel start.
    unsigned long long shared_thr;
};
__device__ __forceinline__ void topk_smem_init(TopkSmem& s) { s.shared_thr = 0ull; }

// Every element of a slice that can belong to the row's top-k: composite
// key >= the filter `theta`.  The filter is only ever raised to a certified
// lower bound on the row's k-th largest key (at least k elements of the row
// reach it), or set from a hint.  With kTies the filter is a value bound
// (low 32 bits zero: every element of the k-th value is kept); without, the
// k-th key is the exact (value desc, index asc) order statistic.
//
// Hints are not certified: the combine verifies them (at least k gathered
// keys reach the filter) and retries the row without a hint otherwise.
// Without a hint, the first chunk's per-thread maxima give the first
// certified bound (they are distinct elements, so the k-th largest of them
// is at most the row's k-th largest).
//
// Candidates are rare, so the hot loop keeps them per thread: a vector
// whose max reaches the filter stores its passing elements in the thread's
// own kSlots slots (no warp synchronisation); a vector that does not fit is
// flagged and re-read at chunk_end(), which also moves the warp's slots into
// the warp's region with one ballot per slot.  A warp whose region fills past half
// raises its own filter to the exact k-th largest of its own candidates
// (again certified) and compacts its region; warps keep their own filters
// and the slice's filter is their maximum.  A region that overflows anyway
// (massive ties with kTies, adversarial order, k above half a region) is
// reported; the combine then takes its exact fallback.
template <class E, bool kTies>
struct TopkHistFn : FnHooks {
    static constexpr bool kPrepass = true;
    static constexpr int VEC = E::kVec;
    static constexpr int kRegion = TopkSmem::kRegion;
    static constexpr int kRefineAt = kRegion / 2;
    TopkSmem* S;
    int k;
    uint64_t theta;     // composite filter, warp-uniform (CTA-uniform until a warp refines)
    float thr_f;        // float prefilter: v >= thr_f  <=>  value key >= hkey(theta)
    float vmx;          // running max with NaN propagation (every element)
    int nw;             // candidates appended by this warp (warp-uniform; may exceed kRegion)
    uint32_t lost;      // this warp's region overflowed
    uint32_t tmax;      // prepass: this thread's max value key
    uint32_t cmask;     // rounds of the current chunk deferred to chunk_end()
    int rr;             // rounds seen in the current chunk
    int tcnt;           // keys in this thread's slots
    uint32_t tag;       // the unit's tag for the shared filter (nonzero, CTA-uniform)

    __device__ __forceinline__ void set_theta(uint64_t t) { theta = t; thr_f = key_to_thr(hkey(t)); }
    // `unit_tag`: nonzero, distinct for every unit a CTA streams
    __device__ __forceinline__ void init(TopkSmem* s, int kk, uint32_t hint, uint32_t unit_tag) {
        S = s; k = kk; tag = unit_tag;
        set_theta(static_cast<uint64_t>(hint) << 32);
        vmx = -kInf; nw = 0; lost = 0; tmax = 0; cmask = 0; rr = 0; tcnt = 0;
    }
    __device__ __forceinline__ bool use_prepass() const { return theta == 0; }
    __device__ __forceinline__ void pre_vec(bool act, const float (&v)[VEC], int) {
        if (!act) return;
        const float m4 = vmax_nan(v);
        if (m4 == m4) tmax = max(tmax, fkey(m4));
    }
    __device__ __forceinline__ void pre_scalar(bool act, float v, int) {
        if (act && v == v) tmax = max(tmax, fkey(v));
    }
    // k-th largest of the warps' top-8 (k <= 64) or top-32 thread maxima (all consumers)
    __device__ void pre_end() {
        const int per = (k <= 8 * kWarps) ? 8 : 32;
        const int P = per * kWarps;
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        const uint64_t srt = warp_sort_desc(static_cast<uint64_t>(tmax));
        if (lane < per) S->pool[w * per + lane] = srt;
        if (threadIdx.x == 0) S->sh64[1] = 0;
        csync();
        if (k <= P && static_cast<int>(threadIdx.x) < P) {
            const uint64_t me = S->pool[threadIdx.x];
            int r = 0, eq = 0;
            for (int t = 0; t < P; ++t) {
                const uint64_t o = S->pool[t];
                r += o > me;
                eq += (o == me) & (t < static_cast<int>(threadIdx.x));
            }
            // the k-th largest value (ties resolved by position)
            if (r + eq == k - 1) S->sh64[1] = me;
        }
        csync();
        const uint64_t b = S->sh64[1] << 32;
        if (b > theta) set_theta(b);
        csync();
    }
    // Append the lanes' candidates (bit j of m: element x + j) to the warp's
    // region: one ballot per element slot, so the positions need no scan.
    __device__ __forceinline__ void append(uint32_t m, const float* v, int x) {
        const uint32_t lt = (1u << (threadIdx.x & 31)) - 1u;
        uint64_t* reg = S->cand + (threadIdx.x >> 5) * kRegion;
        int base = nw;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const bool p = (m >> j) & 1u;
            const uint32_t bj = __ballot_sync(0xffffffffu, p);
            if (p) {
                const int pos = base + __popc(bj & lt);
                if (pos < kRegion) reg[pos] = ckey(v[j], x + j);
            }
            base += __popc(bj);
        }
        nw = base;
    }
    __device__ __forceinline__ bool passes(float v, int x) const {
        return v >= thr_f && (kTies || ckey(v, x) >= theta);
    }
    // Hot loop: the vector max decides whether any element reaches the
    // filter (NaN lands there too; it is never stored).  Passing elements go
    // to the thread's slots, or the round is deferred to chunk_end().
    __device__ __forceinline__ void vec(bool act, const float (&v)[VEC], int x) {
        if (act) {
            const float m4 = vmax_nan(v);
            vmx = max_nan(vmx, m4);
            if (!(m4 < thr_f)) {
                uint32_t m = 0;
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (passes(v[j], x + j)) m |= 1u << j;
                const int c = __popc(m);
                if (tcnt + c <= TopkSmem::kSlots) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        if ((m >> j) & 1u) {
                            S->slot[tcnt][threadIdx.x] = ckey(v[j], x + j);
                            ++tcnt;
                        }
                    }
                } else {
                    cmask |= 1u << rr;
                }
            }
        }
        ++rr;
    }
    // four rounds at once (vector r at x + r * kThreads * VEC): one test
    // whether any element reaches the filter; only then per round as vec()
    static constexpr bool kVec4 = true;
    __device__ __forceinline__ void vec4(const float (&v)[4][VEC], int x) {
        const float m0 = vmax_nan(v[0]), m1 = vmax_nan(v[1]), m2 = vmax_nan(v[2]), m3 = vmax_nan(v[3]);
        const float mm = max_nan(max_nan(m0, m1), max_nan(m2, m3));
        vmx = max_nan(vmx, mm);
        if (!(mm < thr_f)) {
            const float ms[4] = {m0, m1, m2, m3};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (!(ms[r] < thr_f)) {
                    const int xr = x + r * kThreads * VEC;
                    uint32_t m = 0;
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        if (passes(v[r][j], xr + j)) m |= 1u << j;
                    const int c = __popc(m);
                    if (tcnt + c <= TopkSmem::kSlots) {
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            if ((m >> j) & 1u) {
                                S->slot[tcnt][threadIdx.x] = ckey(v[r][j], xr + j);
                                ++tcnt;
                            }
                        }
                    } else {
                        cmask |= 1u << (rr + r);
                    }
                }
            }
        }
        rr += 4;
    }
    __device__ __forceinline__ void scalar(bool act, float v, int x) {
        bool any = false;
        if (act) {
            vmx = max_nan(vmx, v);
            any = passes(v, x);
        }
        if (__any_sync(0xffffffffu, any)) {
            float vv[VEC] = {};
            vv[0] = v;
            append(any ? 1u : 0u, vv, x);
        }
    }
    // per warp: the lanes' slots into the warp's region, one ballot per slot
    __device__ __forceinline__ void flush_slots() {
        if (__any_sync(0xffffffffu, tcnt != 0)) {
            const uint32_t lt = (1u << (threadIdx.x & 31)) - 1u;
            uint64_t* reg = S->cand + (threadIdx.x >> 5) * kRegion;
            int base = nw;
#pragma unroll
            for (int i = 0; i < TopkSmem::kSlots; ++i) {
                const bool p = i < tcnt;
                const uint32_t bal = __ballot_sync(0xffffffffu, p);
                if (p) {
                    const int pos = base + __popc(bal & lt);
                    if (pos < kRegion) reg[pos] = S->slot[i][threadIdx.x];
                }
                base += __popc(bal);
            }
            nw = base;
            tcnt = 0;
        }
    }
    // Before the chunk is released: only the rounds deferred for want of
    // slot room need its data (the slots are flushed after the release).
    __device__ __forceinline__ void chunk_end(int, const unsigned char* sm, int cx0, int nv) {
        if (__any_sync(0xffffffffu, cmask != 0)) {
            for (int r = 0; r < rr; ++r) {
                const bool mine = (cmask >> r) & 1u;
                if (!__any_sync(0xffffffffu, mine)) continue;
                const int vi = r * kThreads + static_cast<int>(threadIdx.x);
                float vals[VEC] = {};
                uint32_t m = 0;
                if (mine && vi < nv) {
                    E::unpack(reinterpret_cast<const uint4*>(sm)[vi], vals);
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        if (passes(vals[j], cx0 + vi * VEC + j)) m |= 1u << j;
                }
                append(m, vals, cx0 + vi * VEC);
                // a filter far below the row's k-th value (a stale hint) passes
                // whole rounds: refine before the region can overflow
                if (nw > kRefineAt) refine_warp();
            }
        }
        cmask = 0;
        rr = 0;
    }
    // per warp, after every chunk: adopt a better filter another warp found;
    // past half a region, refine this warp's own
    __device__ __forceinline__ void after_release(int) {
        const unsigned long long v = *reinterpret_cast<volatile unsigned long long*>(&S->shared_thr);
        if (static_cast<uint32_t>(v >> 32) == tag) {
            const uint64_t t = (v & 0xffffffffull) << 32;
            if (t > theta) set_theta(t);
        }
        // slots are flushed only once a lane's are nearly full (and at the end)
        if (__any_sync(0xffffffffu, tcnt >= TopkSmem::kSlots - 1)) flush_slots();
        if (nw > kRefineAt) refine_warp();
    }
    // A higher filter from this warp's candidates: the value key where at
    // least k of them remain (certified: they are elements of the slice),
    // found by bisection that stops once at most k + k/2 remain; with a
    // bisection that runs to the end and !kTies, the exact k-th composite
    // key.  Then the region is compacted to the keys at or above the filter
    // (keys below a filter another warp raised are dropped too) and the
    // filter is shared with the other warps.
    __device__ void refine_warp() {
        const int lane = threadIdx.x & 31;
        uint64_t* reg = S->cand + (threadIdx.x >> 5) * kRegion;
        const int n = nw < kRegion ? nw : kRegion;
        lost |= nw > kRegion;
        auto count_ge = [&](uint64_t t, bool value_only) {
            int c = 0;
            for (int j0 = 0; j0 < n; j0 += 32) {
                const int j = j0 + lane;
                bool p = false;
                if (j < n) p = value_only ? (hkey(reg[j]) >= static_cast<uint32_t>(t)) : (reg[j] >= t);
                c += __popc(__ballot_sync(0xffffffffu, p));
            }
            return c;
        };
        uint64_t nt = theta;
        int clo = count_ge(hkey(theta), true);
        if (clo >= k) {
            uint32_t mx = 0;
            for (int j = lane; j < n; j += 32) mx = max(mx, hkey(reg[j]));
            uint32_t lo = hkey(theta), hi = warp_max_u32(mx);
            const int enough = k + (k >> 1);
            while (lo < hi && clo > enough) {
                const uint32_t mid = lo + static_cast<uint32_t>((static_cast<uint64_t>(hi) - lo + 1) >> 1);
                const int c = count_ge(mid, true);
                if (c >= k) { lo = mid; clo = c; } else { hi = mid - 1; }
            }
            nt = static_cast<uint64_t>(lo) << 32;
            if (!kTies && clo > enough) {
                // every remaining key shares the value lo: split on the index bits
                uint64_t cl = nt > theta ? nt : theta, ch = nt | 0xffffffffull;
                while (cl < ch) {
                    const uint64_t d = ch - cl;
                    const uint64_t mid = cl + (d >> 1) + (d & 1ull);
                    if (count_ge(mid, false) >= k) cl = mid; else ch = mid - 1;
                }
                nt = cl;
            }
            if (nt > theta) {
                set_theta(nt);
                if (lane == 0)
                    atomicMax(&S->shared_thr, (static_cast<unsigned long long>(tag) << 32) | hkey(nt));
            } else {
                nt = theta;
            }
        }
        const uint32_t lt = (1u << lane) - 1u;
        int out = 0;
        for (int j0 = 0; j0 < n; j0 += 32) {
            const int j = j0 + lane;
            uint64_t key = 0;
            bool p = false;
            if (j < n) { key = reg[j]; p = key >= nt; }
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            if (p) reg[out + __popc(bal & lt)] = key;
            out += __popc(bal);
        }
        nw = out;
        __syncwarp();
    }
    // One-barrier finish, step 1 (per warp): the warp's candidate count,
    // filter, flags (1: a region lost keys, 2: NaN / +inf seen) and max into
    // shared memory.  The caller then csync()s and reads summary().
    __device__ void publish() {
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        flush_slots();
        lost |= nw > kRegion;
        const uint32_t fl = (lost ? 1u : 0u) | (bad_max(vmx) ? 2u : 0u);
        const uint32_t flw = __reduce_or_sync(0xffffffffu, fl);
        float wm = vmx;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wm = max_nan(wm, __shfl_xor_sync(0xffffffffu, wm, o));
        if (lane == 0) {
            S->wn[w] = nw < kRegion ? nw : kRegion;
            S->wthr[w] = theta;
            S->scratch[w] = flw;
            S->wmax[w] = wm;
        }
    }
    // step 2 (every consumer, after the csync): totals over the warps
    __device__ void summary(int& tot, uint64_t& F, uint32_t& flags, float& vm) const {
        tot = 0; F = 0; flags = 0; vm = -kInf;
#pragma unroll
        for (int j = 0; j < kWarps; ++j) {
            tot += S->wn[j];
            F = S->wthr[j] > F ? S->wthr[j] : F;
            flags |= S->scratch[j];
            vm = max_nan(vm, S->wmax[j]);
        }
    }
    // step 3 (per warp): the warp's keys to dst at the warp's offset (the
    // prefix of the warps' counts).  Keys below the slice filter F are kept
    // too: a combine never counts them (it works at or above the largest
    // filter of all slices).
    __device__ void write_keys(uint64_t* dst) const {
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        const uint64_t* reg = S->cand + w * kRegion;
        int base = 0;
        for (int j = 0; j < w; ++j) base += S->wn[j];
        const int n = S->wn[w];
        for (int j = lane; j < n; j += 32) dst[base + j] = reg[j];
    }

    // After the stream (all consumers): the candidates with key >= F (the
    // largest warp filter), compacted to S->cand[0..return).  `oflow` when a
    // region lost keys, `bad` when the slice holds a NaN or +inf, `vm` the
    // slice maximum (NaN-propagating).
    __device__ int finish(uint64_t& F, uint32_t& oflow, uint32_t& bad, float& vm) {
        constexpr int kPer = kRegion / 32;
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        const uint32_t lt = (1u << lane) - 1u;
        flush_slots();
        lost |= nw > kRegion;
        const uint32_t fl = (lost ? 1u : 0u) | (bad_max(vmx) ? 2u : 0u);
        const uint32_t flw = __reduce_or_sync(0xffffffffu, fl);
        float wm = vmx;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wm = max_nan(wm, __shfl_xor_sync(0xffffffffu, wm, o));
        if (lane == 0) { S->wthr[w] = theta; S->scratch[w] = flw; S->wmax[w] = wm; }
        csync();
        F = S->wthr[0];
        uint32_t fa = S->scratch[0];
        vm = S->wmax[0];
#pragma unroll
        for (int j = 1; j < kWarps; ++j) {
            F = S->wthr[j] > F ? S->wthr[j] : F;
            fa |= S->scratch[j];
            vm = max_nan(vm, S->wmax[j]);
        }
        oflow = fa & 1u;
        bad = (fa >> 1) & 1u;
        const uint64_t* reg = S->cand + w * kRegion;
        const int n = nw < kRegion ? nw : kRegion;
        uint64_t key[kPer];
        uint32_t pm = 0;
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int j = i * 32 + lane;
            key[i] = j < n ? reg[j] : 0ull;
            const bool p = j < n && key[i] >= F;
            pm |= static_cast<uint32_t>(p) << i;
            cnt += __popc(__ballot_sync(0xffffffffu, p));
        }
        if (lane == 0) S->ired[w] = cnt;
        csync();   // every warp holds its keys in registers: the regions may be overwritten
        int base = 0, tot = 0;
#pragma unroll
        for (int j = 0; j < kWarps; ++j) {
            const int c = S->ired[j];
            if (j < w) base += c;
            tot += c;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const bool p = (pm >> i) & 1u;
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            if (p) S->cand[base + __popc(bal & lt)] = key[i];
            base += __popc(bal);
        }
        csync();
        return tot;
    }
};

// [p - q]_+ and p weights over one row with known max m and normaliser Z
// (elements below the mask threshold have p = 0: only the -q part, which
// the positive part drops)
template <class E>
struct ResidFn {
    float m, c, invZ;
    float thr = -kInf;
    float r = 0.f, pw = 0.f;
    __device__ __forceinline__ void vec2(bool act, const float (&lv)[E::kVec], const float (&qv)[E::kVec], int) {
        if (!act) return;
#pragma unroll
        for (int j = 0; j < E::kVec; ++j) {
            const float w = lv[j] >= thr ? ex2((lv[j] - m) * c) : 0.f;
            const float d = w * invZ - qv[j];
            r += d > 0.f ? d : 0.f;
            pw += w;
        }
    }
    __device__ __forceinline__ void scalar2(bool act, float l, float q, int) {
        if (!act) return;
        const float w = l >= thr ? ex2((l - m) * c) : 0.f;
        const float d = w * invZ - q;
        r += d > 0.f ? d : 0.f;
        pw += w;
    }
};

// block max of a float with NaN propagation; every thread receives it
__device__ __forceinline__ float block_max_nan(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    csync();
    if (l == 0) red[w] = v;
    csync();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) r = max_nan(r, red[i]);
    return r;
}

}  // namespace spec
