// spec_chain.cu -- batched chain speculative sampling on the row-task engine.
//
// [SD-survey] = "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
// (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash, DDTree and
// DSpark), chzhyang.github.io.  §1 "what speculative decoding guarantees":
// position i accepts its drafted token y_i with probability
// min(1, p_i(y_i)/q_i(y_i)); the first rejection commits a token drawn from
// the normalised residual [p_i - q_i]_+; if every draft passes, a bonus token
// is drawn from p_{K+1}; temperature and top-k truncation are part of p.
//
// Tasks of one request, in order:
//   VERIFY row i   stream logits row i; combine: p_i(y_i), accept test;
//                  accept -> VERIFY i+1 (or BONUS at i = k); reject -> with
//                  top-k the correction is drawn in the same combine (the
//                  residual lives on the top-k set); without top-k -> RESID i
//   RESID row i    (untruncated p only) stream logits row i and q row i
//                  together, sum [p - q]_+ per slice, then draw the token
//   BONUS row k    stream logits row k, draw from p
// Rows past the first rejection are never touched.
#include "spec_chain.cuh"
#include "spec_select.cuh"

namespace spec {

enum ChainKind : int { kVerify = 0, kBonus = 1, kResid = 2, kInvalid = 3 };
constexpr int kKindMask = 7;
constexpr int kNoHint = 8;        // kind bit: stream the row without a filter hint (a retry)

// Combiner scratch: the gathered candidate keys, then the top-k set sorted by
// token (ids and fp64 weights; a larger tied set takes the exact fallback).
constexpr int kCombKeys = 2048;
constexpr int kCombSet = 512;
// A top-k combine as the combiner warp prepared it for the consumers: the
// gathered keys are in CombSmem::list.
struct CombPrep {
    int b, row, kind, st;
    int n;            // gathered keys
    int y;            // drafted token (VERIFY)
    int fallback;     // 1: a slice overflowed; take the exact path
    int hinted;       // a slice streamed behind a hint
    int sl;           // slice length of the row
    uint32_t done;    // finished requests when the row arrived (an estimate, for the next row's slicing)
    uint32_t base;    // arrival base of the request's next task
    float vmax;
    float pad;
    uint64_t theta;   // largest slice filter
    float uk, ur;     // uniforms: sample, accept
    // an untruncated draw: rescan slice [x0, x1) for the CDF crossing t
    int x0, x1, wmode;  // wmode 0: p weights 2^((l-m)c); 1: [p - q]_+
    float m, invZf;
    dfloat t;
    double Z, R;        // diagnostics
};
// Written by the combiner warp while the consumers stream; the consumers'
// own scratch for a combine lives in TopkSmem (free at unit boundaries,
// where they serve combines): select ranks in `slot`, the selected keys in
// the first kCombOut entries of `cand`, tokens and weights after them.
struct CombSmem {
    SliceHdrs hdrs;
    CombPrep prep;
    alignas(16) uint64_t list[kCombKeys];
};
constexpr int kCombOut = 1024;   // select output (> kCombSet: a larger set takes the exact path)
static_assert(sizeof(uint64_t) * TopkSmem::kSlots * kThreads >= sizeof(int) * kCombKeys, "ranks fit in slot");
static_assert(sizeof(uint64_t) * (kCombOut) + (sizeof(int) + sizeof(float2)) * kCombSet <=
                  sizeof(uint64_t) * kWarps * TopkSmem::kRegion,
              "selected keys, tokens and weights fit in cand");

template <bool kTopk> struct ChainTopkPart {};
template <> struct ChainTopkPart<true> { TopkSmem tk; };

template <bool kTopk>
struct __align__(16) ChainSmem : ChainTopkPart<kTopk> {
    PipeSmem pipe;
    CombSmem comb;
    uint64_t sh64[4];
    int ish[4];
    float2 red2[kWarps];
    int ired[kWarps + 4];
    int hist[64];
    uint32_t scratch[kWarps + 2];
    float fsh[8];
    float wm[kWarps];        // per-warp partials of the one-barrier finishes
    float2 ws[kWarps];       // float-float
    float2 ws2[kWarps];
    uint32_t wb[kWarps];
};

__device__ __forceinline__ int chain_k(const ChainArgs& A, int b) {
    return A.k_per_req ? A.k_per_req[b] : A.K;
}
template <class E>
__device__ __forceinline__ const void* chain_lrow(const ChainArgs& A, int b, int i) {
    const long long r = A.k_per_req ? static_cast<long long>(A.l_row_off[b] + i) * A.l_rs
                                    : static_cast<long long>(b) * A.l_bs + static_cast<long long>(i) * A.l_rs;
    return static_cast<const unsigned char*>(A.logits) + r * E::kBytes;
}
__device__ __forceinline__ const float* chain_qrow(const ChainArgs& A, int b, int i) {
    const long long r = A.k_per_req ? static_cast<long long>(A.q_row_off[b] + i) * A.q_rs
                                    : static_cast<long long>(b) * A.q_bs + static_cast<long long>(i) * A.q_rs;
    return A.q + r;
}
__device__ __forceinline__ float chain_u(const ChainArgs& A, int b, int i) {
    return A.uniforms[static_cast<long long>(b) * (A.K + 1) + i];
}

// ---------------------------------------------------------------------------
// combiner-warp steps (all 32 lanes unless stated)
// ---------------------------------------------------------------------------
// Commit the request: accepted drafts, then `last` (correction/bonus, or -1),
// then -1 padding; lane 0 publishes completion.
__device__ void chain_finish(const ChainArgs& A, int b, int n, int last, int st) {
    const int W = A.K + 1;
    int* out = A.out_tokens + static_cast<long long>(b) * W;
    for (int i = threadIdx.x & 31; i < W; i += 32) {
        int v = -1;
        if (i < n) v = A.draft[static_cast<long long>(b) * A.K + i];
        else if (i == n) v = last;
        out[i] = v;
    }
    if ((threadIdx.x & 31) == 0) {
        A.num_accepted[b] = n;
        A.status[b] = st;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) finish_request(A.W);
}

// The same on every consumer thread (a combine the consumers run).
__device__ void chain_finish_cta(const ChainArgs& A, int b, int n, int last, int st) {
    const int W = A.K + 1;
    int* out = A.out_tokens + static_cast<long long>(b) * W;
    for (int i = threadIdx.x; i < W; i += kThreads) {
        int v = -1;
        if (i < n) v = A.draft[static_cast<long long>(b) * A.K + i];
        else if (i == n) v = last;
        out[i] = v;
    }
    if (threadIdx.x == 0) {
        A.num_accepted[b] = n;
        A.status[b] = st;
    }
    csync();
    if (threadIdx.x == 0) finish_request(A.W);
}

__device__ __forceinline__ void chain_diag(const ChainArgs& A, int b, int i, float py, float qy, float Z, float R) {
    if (!A.diag) return;
    float* d = A.diag + (static_cast<long long>(b) * (A.K + 1) + i) * 4;
    d[0] = py; d[1] = qy; d[2] = Z; d[3] = R;
}

// lane 0: push the request's next task after an accepted position (the
// record carries all the task needs: no release)
__device__ void chain_advance(const ChainArgs& A, int b, int row, int kb, int st, uint32_t hint, uint32_t done,
                              uint32_t base) {
    Task t;
    t.b = b;
    t.row = row + 1;
    t.kind = (row + 1 < kb) ? kVerify : kBonus;
    t.aux = static_cast<int>(hint);
    t.st = st;
    t.base = base;
    int S, SL;
    pick_slices(A.B, A.V, A.S, A.S1, done, S, SL);
    push_task(A.W, t, S, SL, false);
}

// Acceptance of drafted y: u < p(y)/q(y).  With weights scaled by the
// normaliser, p(y) = e_y / Z, the test is e_y > u q Z (float-float; no
// division on this path).  A ratio within rounding of u is a near tie.
__device__ __forceinline__ bool chain_accept_z(const ChainArgs& A, int y, float ey, float qy, dfloat Z, float u,
                                               int& st) {
    if (y < 0 || y >= A.V) {
        st |= 8;
        return false;
    }
    if (qy == 0.f) {
        st |= 2;
        return ey > 0.f;   // p/q = inf when p > 0, else 0
    }
    return df_gt(df_make(ey), df_mul(u, df_mul(qy, Z)));
}

// Inverse CDF over n (token, weight) pairs sorted by token, float-float
// weights; the smallest token with prefix > t.  Result in every lane.
__device__ int warp_icdf_pairs(const int* tok, const float2* w, int n, dfloat t) {
    const int lane = threadIdx.x & 31;
    const int per = (n + 31) / 32;
    const int i0 = lane * per, i1 = min(n, i0 + per);
    dfloat loc = df_make(0.f);
    for (int i = i0; i < i1; ++i) loc = df_add(loc, dfloat{w[i].x, w[i].y});
    dfloat tot;
    dfloat c = warp_exscan_df(loc, tot);
    int found = 0x7fffffff, lastpos = -1;
    for (int i = i0; i < i1; ++i) {
        if (w[i].x > 0.f) {
            lastpos = i;
            c = df_add(c, dfloat{w[i].x, w[i].y});
            if (df_gt(c, t) && found == 0x7fffffff) found = i;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
        lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
    }
    const int pick = found != 0x7fffffff ? found : (lastpos >= 0 ? lastpos : 0);
    return n > 0 ? tok[pick] : -1;
}

// Filter hint for the next row from this row's top-k threshold tau and max
// m: 0.15 of the gap below tau (rows of one target differ little in tau; a
// hint above the next row's tau only costs a re-read of that row).
#ifndef SPEC_HINT_MARGIN
#define SPEC_HINT_MARGIN 0.15f
#endif
__device__ __forceinline__ uint32_t next_hint(float tau, float m) {
    const float h = tau - SPEC_HINT_MARGIN * (m - tau);
    return (h == h && h > -kInf) ? fkey(h) : 0u;
}

// ---------------------------------------------------------------------------
// combine with top-k: the candidate lists of all slices hold S exactly
// ---------------------------------------------------------------------------
// Combiner warp, last arrival of a top-k row: everything that waits on
// global memory -- the slice headers, the drafted token, the uniforms, every
// slice key -- into shared memory for the consumers.  Returns false when the
// combine ended here (a bad row).
template <class E>
__device__ bool prepare_topk(const ChainArgs& A, CombSmem& cs, int b, int row, int kind, int st, int S, int SL,
                             uint32_t done, uint32_t base) {
    const int l = threadIdx.x & 31;
    const int kb = chain_k(A, b);
    const float uk = chain_u(A, b, kb);
    const float ur = kind == kVerify ? chain_u(A, b, row) : 0.f;
    const int y = kind == kVerify ? A.draft[static_cast<long long>(b) * A.K + row] : -1;
    SliceHdrs& H = cs.hdrs;
    const int pre = load_hdrs_w(A.W, b, S, H, cs.list, kCombKeys);   // headers and each slice's first keys
    SPEC_TRACE_EVW(5, b, row, S, kind);
    uint32_t flags = 0;
    float vmax = -kInf;
    uint64_t theta = 0;
    if (l < S) { flags = H.flags[l]; vmax = H.vmax[l]; theta = H.kth[l]; }
    flags = __reduce_or_sync(0xffffffffu, flags);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        vmax = max_nan(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        const uint64_t t2 = __shfl_xor_sync(0xffffffffu, theta, o);
        theta = t2 > theta ? t2 : theta;
    }
    if ((flags & kPfBad) || !(vmax > -kInf)) {
        chain_finish(A, b, row, -1, st | 1);
        return false;
    }
    int n = 0, fb = (flags & kPfOverflow) ? 1 : 0;
    if (!fb) {
        bool oflow;
        n = gather_all_w(A.W, b, S, H, cs.list, kCombKeys, oflow, pre);
        if (oflow) fb = 1;
    }
    SPEC_TRACE_EVW(6, b, row, n, kind);
    if (l == 0) {
        CombPrep& p = cs.prep;
        p.b = b; p.row = row; p.kind = kind; p.st = st; p.n = n; p.y = y; p.fallback = fb;
        p.sl = SL;
        p.done = done;
        p.base = base;
        p.hinted = (flags & kPfHinted) ? 1 : 0;
        p.vmax = vmax; p.theta = theta; p.uk = uk; p.ur = ur;
    }
    return true;
}

template <class E>
__device__ void chain_fallback_cta(const ChainArgs& A, ChainSmem<true>& sh, int b, int row, int kind,
                                   int st, float vmax);

// Consumers: the compute of a prepared top-k combine.  The set S of the
// row's k largest values (ties kept) from the gathered keys, its normaliser
// Z, then the accept test at the drafted token, or a draw from the residual
// [p - q]_+ on S (rejection) or from p (bonus row).
template <class E>
__device__ void combine_topk_cta(const ChainArgs& A, ChainSmem<true>& sh) {
    CombSmem& cs = sh.comb;
    const CombPrep p = cs.prep;
    const int b = p.b, row = p.row, kind = p.kind, k = A.top_k;
    int st = p.st;
    SPEC_TRACE_EV(20, b, row, 0, kind);
    const int kb = chain_k(A, b);
    if (p.fallback) {
        chain_fallback_cta<E>(A, sh, b, row, kind, st, p.vmax);
        return;
    }
    uint64_t* list = cs.list;
    const uint32_t th = hkey(p.theta);
    // keys at or above the largest slice filter: enough for the k-th?
    int n = compact_list(list, p.n, th, sh.ired);
    if (n < k) {
        if (p.hinted) {
            // the hint was above the row's k-th value: stream the row again without it
            if (threadIdx.x == 0) {
                Task t;
                t.b = b; t.row = row; t.kind = kind | kNoHint; t.aux = 0; t.st = st; t.base = p.base;
                int S, SL;
                pick_slices(A.B, A.V, A.S, A.S1, p.done, S, SL);
                push_task(A.W, t, S, SL, false);
            }
            return;
        }
        chain_fallback_cta<E>(A, sh, b, row, kind, st, p.vmax);
        return;
    }
    uint64_t kth;
    bool of = false;
    uint64_t* cand = sh.tk.cand;
    int* ctok = reinterpret_cast<int*>(cand + kCombOut);
    float2* cwgt = reinterpret_cast<float2*>(ctok + kCombSet);
    const int keep = select_to(list, n, k, true, reinterpret_cast<int*>(&sh.tk.slot[0][0]), cand, kCombOut, kth, of,
                               sh.sh64, sh.ired);
    SPEC_TRACE_EV(7, b, row, n, kind);
    if (of || keep > kCombSet) {
        chain_fallback_cta<E>(A, sh, b, row, kind, st, p.vmax);
        return;
    }
    // S = cand[0 .. keep): values >= tau, sorted by value descending
    const uint32_t tau_key = hkey(cand[keep - 1]);
    const float tau = ckey_val(cand[keep - 1]);
    // weights e_x = 2^((l_x - m) c) and Z = sum over S in float-float; p(x) =
    // e_x / Z is never formed on this path (tests compare Z-scaled masses)
    // Each thread holds up to kPer members of S: token, weight, and (VERIFY)
    // q at the token, loaded now so that a rejection finds it in registers.
    constexpr int kPer = kCombSet / kThreads;
    const float m = p.vmax, c2 = A.c2;
    const float* qrow = kind == kVerify ? chain_qrow(A, b, row) : nullptr;
    int xs[kPer];
    float ev[kPer], qv[kPer];
    dfloat zpart = df_make(0.f);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int i = threadIdx.x + j * kThreads;
        xs[j] = -1; ev[j] = 0.f; qv[j] = 0.f;
        if (i < keep) {
            xs[j] = ckey_idx(cand[i]);
            ev[j] = ex2((ckey_val(cand[i]) - m) * c2);
            zpart = df_add(zpart, ev[j]);
            if (qrow && xs[j] >= 0 && xs[j] < A.V) qv[j] = __ldcg(qrow + xs[j]);   // keys hold in-range ids
        }
    }
    const dfloat Z = block_sum_df(zpart, sh.red2);
    const float Zf = Z.hi;
    auto prob = [&](float e) { return static_cast<float>(static_cast<double>(e) / df_to_d(Z)); };   // diagnostics
    const uint32_t hint = next_hint(tau, m);
    SPEC_TRACE_EV(8, b, row, keep, kind);
    if (threadIdx.x == 0) {
        __stcg(&A.W.ctrl->hint0, hint);
        // for the next call's first rows: a wider margin (another call's rows
        // may sit lower)
        const float hw = tau - 0.5f * (m - tau);
        __stcg(&A.W.persist[1], (hw == hw && hw > -kInf) ? fkey(hw) : 0u);
        __stcg(&A.W.persist[2], static_cast<uint32_t>(A.V));
        __stcg(&A.W.persist[3], static_cast<uint32_t>(A.top_k));
        __stcg(&A.W.persist[0], kPersistTag);
    }

    // Z-scaled weights of S sorted by token id (ascending): e_x, or for the
    // residual Z [p - q]_+ = [e_x - q_x Z]_+
    int rk[kPer];
    bool ranked = false;
    auto sort_by_token = [&](bool residual, dfloat& total) {
        if (!ranked) {
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                rk[j] = 0;
                if (threadIdx.x + j * kThreads < keep)
                    for (int t = 0; t < keep; ++t) rk[j] += ckey_idx(cand[t]) < xs[j];   // ids in S are distinct
            }
            ranked = true;
        }
        dfloat part = df_make(0.f);
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (threadIdx.x + j * kThreads >= keep) continue;
            dfloat w = df_make(ev[j]);
            if (residual) {
                const dfloat d = df_add(w, df_neg(df_mul(qv[j], Z)));
                w = d.hi > 0.f ? d : df_make(0.f);
            }
            ctok[rk[j]] = xs[j];
            cwgt[rk[j]] = make_float2(w.hi, w.lo);
            part = df_add(part, w);
        }
        total = block_sum_df(part, sh.red2);
    };

    if (kind == kVerify) {
        const int y = p.y;
        float ey = 0.f, qy = 0.f;
        if (y >= 0 && y < A.V) {
            const int sy = y / p.sl;
            const float ly = cs.hdrs.ly[sy];
            qy = cs.hdrs.qy[sy];
            if (fkey(ly) >= tau_key) ey = ex2((ly - m) * c2);
        }
        const bool acc = chain_accept_z(A, y, ey, qy, Z, p.ur, st);
        if (acc) {
            if (threadIdx.x == 0) {
                if (A.diag) chain_diag(A, b, row, prob(ey), qy, Zf, 0.f);
                chain_advance(A, b, row, kb, st, hint, p.done, p.base);
            }
            SPEC_TRACE_EV(9, b, row, 1, kind);
            return;
        }
        // residual [p - q]_+ lives on S (p = 0 outside it)
        dfloat R_mass;
        sort_by_token(true, R_mass);
        if (!(R_mass.hi > 0.f)) {
            st |= 4;
            sort_by_token(false, R_mass);
        }
        int x = -1;
        if (threadIdx.x < 32)
            x = warp_icdf_pairs(ctok, cwgt, keep, df_mul(p.uk, R_mass));
        if (threadIdx.x == 0) {
            sh.ish[0] = x;
            if (A.diag) chain_diag(A, b, row, prob(ey), qy, Zf, (st & 4) ? 0.f : static_cast<float>(df_to_d(R_mass) / df_to_d(Z)));
        }
        csync();
        SPEC_TRACE_EV(11, b, row, 0, kind);
        chain_finish_cta(A, b, row, sh.ish[0], st);
        SPEC_TRACE_EV(9, b, row, 0, kind);
        return;
    }
    // bonus row: draw from p
    dfloat tot;
    sort_by_token(false, tot);
    int x = -1;
    if (threadIdx.x < 32) x = warp_icdf_pairs(ctok, cwgt, keep, df_mul(p.uk, tot));
    if (threadIdx.x == 0) sh.ish[0] = x;
    csync();
    x = sh.ish[0];
    if (threadIdx.x == 0 && A.diag && x >= 0 && x < A.V)
        chain_diag(A, b, row, prob(ex2((E::load(chain_lrow<E>(A, b, row), x) - m) * c2)), 0.f, Zf, 0.f);
    chain_finish_cta(A, b, row, x, st);
}

// Exact path for rows whose top-k set did not fit the candidate buffers
// (massive ties, adversarial order), on the consumers: tau by bisection over
// order-preserving keys, then full-row passes.  Slow; correctness only.
template <class E>
__device__ void chain_fallback_cta(const ChainArgs& A, ChainSmem<true>& sh, int b, int row, int kind,
                                   int st, float vmax) {
    const void* lrow = chain_lrow<E>(A, b, row);
    const int V = A.V, k = A.top_k;
    // largest key t with #{x : key(l_x) >= t} >= k
    // invariant: count(lo) >= k (count(0) = V > k); the range halves every
    // step (64-bit midpoint: hi - lo + 1 can be 2^32), so 32 steps suffice
    uint32_t lo = 0, hi = 0xffffffffu;
    for (int it = 0; it < 33 && lo < hi; ++it) {
        const uint32_t mid = lo + static_cast<uint32_t>((static_cast<uint64_t>(hi) - lo + 1) >> 1);
        int c = 0;
        for (int x = threadIdx.x; x < V; x += kThreads) c += fkey(E::load(lrow, x)) >= mid;
        c = block_sum_i(c, sh.ired);
        if (c >= k) lo = mid; else hi = mid - 1;
    }
    const uint32_t tau = lo;
    const float m = vmax, c2 = A.c2;
    auto wp = [&](int x) -> float {
        const float v = E::load(lrow, x);
        return fkey(v) >= tau ? ex2((v - m) * c2) : 0.f;
    };
    // Z-scaled weights, as in the candidate-set combine
    const dfloat Z = cta_sum(0, V, wp, sh.red2);
    const double Zd = df_to_d(Z);
    const int kb = chain_k(A, b);
    const float uk = chain_u(A, b, kb);
    if (kind == kVerify) {
        const int y = A.draft[static_cast<long long>(b) * A.K + row];
        float ey = 0.f, qy = 0.f;
        if (y >= 0 && y < V) {
            ey = wp(y);
            qy = chain_qrow(A, b, row)[y];
        }
        auto py = [&]() { return static_cast<float>(static_cast<double>(ey) / Zd); };   // diagnostics
        if (chain_accept_z(A, y, ey, qy, Z, chain_u(A, b, row), st)) {
            if (threadIdx.x == 0) {
                if (A.diag) chain_diag(A, b, row, py(), qy, Z.hi, 0.f);
                chain_advance(A, b, row, kb, st, 0u, sh.comb.prep.done, sh.comb.prep.base);
            }
            return;
        }
        const float* qrow = chain_qrow(A, b, row);
        auto wr = [&](int x) -> float {   // Z [p - q]_+
            const dfloat d = df_add(df_make(wp(x)), df_neg(df_mul(qrow[x], Z)));
            return d.hi > 0.f ? d.hi : 0.f;
        };
        const dfloat R_mass = cta_sum(0, V, wr, sh.red2);
        int x;
        if (R_mass.hi > 0.f) {
            x = cta_icdf(0, V, df_mul(uk, R_mass), wr, sh.red2, sh.ired);
        } else {
            st |= 4;
            x = cta_icdf(0, V, df_mul(uk, Z), wp, sh.red2, sh.ired);
        }
        if (threadIdx.x == 0 && A.diag)
            chain_diag(A, b, row, py(), qy, Z.hi, (st & 4) ? 0.f : static_cast<float>(df_to_d(R_mass) / Zd));
        chain_finish_cta(A, b, row, x, st);
        return;
    }
    const int x = cta_icdf(0, V, df_mul(uk, Z), wp, sh.red2, sh.ired);
    if (threadIdx.x == 0 && A.diag && x >= 0 && x < V)
        chain_diag(A, b, row, static_cast<float>(static_cast<double>(wp(x)) / Zd), 0.f, Z.hi, 0.f);
    chain_finish_cta(A, b, row, x, st);
}

// ---------------------------------------------------------------------------
// combine without truncation: per-slice (max, sum of 2^((l-m_s)c))
// ---------------------------------------------------------------------------
// the slice whose running prefix of v (lane s holds slice s's value) crosses
// t, and the prefix before it (float-float)
__device__ __forceinline__ int find_slice_w(int S, dfloat v, dfloat t, dfloat& before) {
    const int l = threadIdx.x & 31;
    if (l >= S) v = df_make(0.f);
    dfloat tot;
    const dfloat ex = warp_exscan_df(v, tot);
    const uint32_t bal = __ballot_sync(0xffffffffu, v.hi > 0.f && df_gt(df_add(ex, v), t));
    int pick;
    if (bal) {
        pick = __ffs(bal) - 1;
    } else {
        const uint32_t pos = __ballot_sync(0xffffffffu, v.hi > 0.f);
        pick = pos ? 31 - __clz(pos) : 0;
    }
    before.hi = __shfl_sync(0xffffffffu, ex.hi, pick);
    before.lo = __shfl_sync(0xffffffffu, ex.lo, pick);
    return pick;
}

__device__ __forceinline__ dfloat df_of(float2 v) { return dfloat{v.x, v.y}; }

// Combiner warp: the combine of an untruncated row.  Returns true when a draw
// needs a slice rescan, prepared in cs.prep for the consumers.  Slice sums
// are Z-scaled (weights e_x = 2^((l_x - m) c)), float-float across slices.
template <class E>
__device__ bool combine_full(const ChainArgs& A, CombSmem& cs, int b, int row, int kind, int st, int S, int SL,
                             uint32_t done, uint32_t base) {
    const int l = threadIdx.x & 31;
    const int kb = chain_k(A, b);
    const float c2 = A.c2;
    const float uk = chain_u(A, b, kb);
    const float ur = kind == kVerify ? chain_u(A, b, row) : 0.f;
    const int y = kind == kVerify ? A.draft[static_cast<long long>(b) * A.K + row] : -1;
    SliceHdrs& H = cs.hdrs;
    load_hdrs_w(A.W, b, S, H);
    SPEC_TRACE_EVW(5, b, row, S, kind);
    if (kind == kResid) {
        const ReqState* rs = &A.W.req[b];
        const dfloat rv = l < S ? df_of(H.sum[l]) : df_make(0.f);
        const dfloat pv = l < S ? df_of(H.sum2[l]) : df_make(0.f);
        const dfloat R_mass = warp_sum_df(rv);
        const dfloat P_mass = warp_sum_df(pv);
        dfloat before, t;
        int s, wmode;
        if (R_mass.hi > 0.f) {
            t = df_mul(uk, R_mass);
            s = find_slice_w(S, rv, t, before);
            wmode = 1;
        } else {
            st |= 4;
            t = df_mul(uk, P_mass);
            s = find_slice_w(S, pv, t, before);
            wmode = 0;
        }
        if (l == 0) {
            CombPrep& p = cs.prep;
            p.b = b; p.row = row; p.kind = kind; p.st = st;
            p.x0 = s * SL; p.x1 = min(A.V, p.x0 + SL); p.wmode = wmode;
            p.m = __ldcg(&rs->m); p.invZf = __ldcg(&rs->invZ);
            p.t = df_add(t, df_neg(before));
            p.Z = 0.0;
            p.R = df_to_d(R_mass);
        }
        return true;   // the consumers rescan the slice
    }
    // VERIFY or BONUS: max and normaliser from the slice partials
    uint32_t flags = l < S ? H.flags[l] : 0u;
    float vmax = l < S ? H.vmax[l] : -kInf;
    flags = __reduce_or_sync(0xffffffffu, flags);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vmax = max_nan(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    if ((flags & kPfBad) || !(vmax > -kInf)) {
        chain_finish(A, b, row, -1, st | 1);
        return false;
    }
    const float m = vmax;
    dfloat zv = df_make(0.f);
    if (l < S && H.sum[l].x > 0.f) zv = df_mul(ex2((H.vmax[l] - m) * c2), df_of(H.sum[l]));
    const dfloat Z = warp_sum_df(zv);
    if (kind == kVerify) {
        float ey = 0.f, qy = 0.f;
        if (y >= 0 && y < A.V) {
            const int sy = y / SL;
            ey = ex2((H.ly[sy] - m) * c2);
            qy = H.qy[sy];
        }
        const bool acc = chain_accept_z(A, y, ey, qy, Z, ur, st);
        if (l == 0 && A.diag) chain_diag(A, b, row, static_cast<float>(static_cast<double>(ey) / df_to_d(Z)), qy, Z.hi, 0.f);
        if (acc) {
            if (l == 0) chain_advance(A, b, row, kb, st, 0u, done, base);
            return false;
        }
        if (l == 0) {
            ReqState* rs = &A.W.req[b];
            __stcg(&rs->m, m);
            __stcg(&rs->invZ, __frcp_rn(Z.hi));
            Task t;
            t.b = b; t.row = row; t.kind = kResid; t.aux = 0; t.st = st; t.base = base;
            int S1, SL1;
            pick_slices(A.B, A.V, A.S, A.S1, done, S1, SL1);
            push_task(A.W, t, S1, SL1, true);   // the residual units read m and 1/Z
        }
        return false;
    }
    // BONUS: inverse CDF of p; find the slice, the consumers rescan it
    const dfloat t = df_mul(uk, Z);
    dfloat before;
    const int s = find_slice_w(S, zv, t, before);
    if (l == 0) {
        CombPrep& p = cs.prep;
        p.b = b; p.row = row; p.kind = kind; p.st = st;
        p.x0 = s * SL; p.x1 = min(A.V, p.x0 + SL); p.wmode = 0;
        p.m = vmax; p.invZf = 0.f;
        p.t = df_add(t, df_neg(before));
        p.Z = df_to_d(Z); p.R = 0.0;
    }
    return true;
}

// Consumers: the rescan of an untruncated draw prepared by combine_full --
// the inverse CDF over one slice -- then the commit.
template <class E>
__device__ void rescan_cta(const ChainArgs& A, ChainSmem<false>& sh) {
    const CombPrep p = sh.comb.prep;
    const int b = p.b, row = p.row;
    const void* lrow = chain_lrow<E>(A, b, row);
    const float m = p.m, c2 = A.c2, invZ = p.invZf;
    int x;
    if (p.wmode == 1) {
        const float* qrow = chain_qrow(A, b, row);
        auto wr = [&](int xx) -> float {
            const float d = ex2((E::load(lrow, xx) - m) * c2) * invZ - qrow[xx];
            return d > 0.f ? d : 0.f;
        };
        x = cta_icdf(p.x0, p.x1, p.t, wr, sh.red2, sh.ired);
    } else {
        auto wp = [&](int xx) -> float { return ex2((E::load(lrow, xx) - m) * c2); };
        x = cta_icdf(p.x0, p.x1, p.t, wp, sh.red2, sh.ired);
    }
    if (threadIdx.x == 0) {
        if (p.kind == kResid) {
            if (A.diag) A.diag[(static_cast<long long>(b) * (A.K + 1) + row) * 4 + 3] = (p.st & 4) ? 0.f : (float)p.R;
        } else if (A.diag && x >= 0 && x < A.V) {
            chain_diag(A, b, row, static_cast<float>(static_cast<double>(ex2((E::load(lrow, x) - m) * c2)) / p.Z), 0.f,
                       static_cast<float>(p.Z), 0.f);
        }
    }
    chain_finish_cta(A, b, row, x, p.st);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// what a unit streams: logits row range (VERIFY/BONUS), logits and q
// (RESID), nothing (invalid k)
template <class E>
__device__ __forceinline__ int chain_unit_kind(const ChainArgs& A, const Task& t) {
    if (t.kind >= 0) return t.kind & kKindMask;
    const int kb = chain_k(A, t.b);
    return (kb < 0 || kb > A.K) ? kInvalid : (kb == 0 ? kBonus : kVerify);
}
template <class E>
__device__ __forceinline__ StreamPlan chain_plan(const ChainArgs& A, const Task& t, int kind, int slice) {
    const int SL = task_SL(A, t);
    const int x0 = slice * SL, x1 = min(A.V, x0 + SL);
    if (kind == kVerify || kind == kBonus) return plan_single(chain_lrow<E>(A, t.b, t.row), E::kBytes, x0, x1);
    if (kind == kResid) return plan_dual(chain_lrow<E>(A, t.b, t.row), E::kBytes, chain_qrow(A, t.b, t.row), x0, x1);
    return plan_none();
}

template <class E, bool kTopk>
__global__ void __launch_bounds__(kBlockThreads, kCtasPerSm) chain_kernel(const ChainArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    auto& sh = *reinterpret_cast<ChainSmem<kTopk>*>(smem + kStages * kChunkBytes);
    if constexpr (kTopk) {
        if (threadIdx.x == 0) topk_smem_init(sh.tk);   // made visible by pipe_init's barrier
    }
    const Pipe P = pipe_init(smem, sh.pipe);
    // the residual pass streams q beside the logits; without q rows (K = 0)
    // there is no residual pass
    const bool tma = A.tma_l && (kTopk || A.K == 0 || A.tma_q);
    if (threadIdx.x >= kCombiner0) {
        // combiner warp: arrivals, combines (top-k: prepared here, computed by
        // the consumers at their next wait)
        uint32_t cpub = 0;
        combiner_loop(P, [&](const Job& job) {
            const int b = job.task.b;
            uint32_t done, base;
            if (!comb_arrive(A.W, job.task, task_S(A, job.task), &done, &base)) return;
            SPEC_TRACE_EVW(2, b, job.task.row, job.slice, job.kind);
            const int st = job.task.st;
            if (job.kind == kInvalid) {
                chain_finish(A, b, 0, -1, 16);
            } else if (!combine_reuse(P, cpub)) {
                return;   // the consumers stopped answering: the kernel is aborting
            } else if constexpr (kTopk) {
                if (prepare_topk<E>(A, sh.comb, b, job.task.row, job.kind, st, task_S(A, job.task),
                                    task_SL(A, job.task), done, base))
                    publish_combine(P, cpub);
            } else {
                if (combine_full<E>(A, sh.comb, b, job.task.row, job.kind, st, task_S(A, job.task),
                                    task_SL(A, job.task), done, base))
                    publish_combine(P, cpub);
            }
            __syncwarp();
            SPEC_TRACE_EVW(3, b, job.task.row, job.slice, job.kind);
        }, [&]() { combine_reuse(P, cpub); });
        return;
    }
    if (threadIdx.x >= kThreads) {
        if (threadIdx.x == kProducer) {
            producer_loop(A.W, A.B, A.S, P, tma,
                          [&](Claimed& c) {
                              if (kTopk && c.task.kind < 0) {
                                  // the latest finished row of this call, else of the previous call
                                  // on this workspace (all five words in one round trip)
                                  const uint32_t h0 = __ldcg(&A.W.ctrl->hint0);
                                  const uint4 ps = __ldcg(reinterpret_cast<const uint4*>(A.W.persist));
                                  c.hint = h0;
                                  if (h0 == 0 && ps.x == kPersistTag && ps.z == static_cast<uint32_t>(A.V) &&
                                      ps.w == static_cast<uint32_t>(A.top_k))
                                      c.hint = ps.y;
                              }
                          },
                          [&](const Claimed& c) {
                              return chain_plan<E>(A, c.task, chain_unit_kind<E>(A, c.task), c.slice);
                          });
        }
        return;
    }
    uint32_t seq = 0, jseq = 0, cseq = 0;
    auto serve = [&]() {
        if constexpr (kTopk) combine_topk_cta<E>(A, sh);
        else rescan_cta<E>(A, sh);
    };
    for (uint32_t u = 0;; ++u) {
        const Claimed cl = next_unit(P, u, cseq, serve);
        if (!cl.ok) break;
        const Task t = cl.task;
        const int s = cl.slice;
        SPEC_TRACE_EV(0, t.b, t.row, s, t.kind);
        const int b = t.b;
        const int row = t.row;
        const bool initial = t.kind < 0;
        const int kind = chain_unit_kind<E>(A, t);
        const bool nohint = !initial && (t.kind & kNoHint);
        PartHdr* ph = part_hdr(A.W, b, s, A.S);
        uint64_t* pk = part_keys(A.W, b, s, A.S);
        const int SLt = task_SL(A, t);
        const int x0 = s * SLt, x1 = min(A.V, x0 + SLt);
        const StreamPlan plan = chain_plan<E>(A, t, kind, s);
        bool ok = true;
        if (kind == kVerify || kind == kBonus) {
            // the drafted token: its logit is recorded as the slice streams,
            // its q fetched early by the slice that holds it
            DraftWatch dw;
            dw.x0 = x0; dw.x1 = x1;
            if (kind == kVerify) {
                dw.y = A.draft[static_cast<long long>(b) * A.K + row];
                dw.qrow = chain_qrow(A, b, row);
            }
            float* wsl = sh.fsh;
            if constexpr (kTopk) {
                const uint32_t hint = nohint ? 0u : (initial ? cl.hint : static_cast<uint32_t>(t.aux));
                TopkHistFn<E, true> fn;
                fn.init(&sh.tk, A.top_k, hint, u + 1u);
                fn.dw = dw;
                ok = consume_row<E>(P, seq, plan, tma, x0, fn);
                if (ok) {
                    SPEC_TRACE_EV(4, b, row, s, kind);
                    fn.publish();
                    if (fn.dw.seen) wsl[0] = fn.dw.ly;
                    csync();
                    int tot;
                    uint64_t F;
                    uint32_t fl;
                    float vm;
                    fn.summary(tot, F, fl, vm);
                    const uint32_t bad = (fl >> 1) & 1u;
                    uint32_t oflow = fl & 1u;
                    int n = tot;
                    if (!bad && !oflow && tot <= A.cap_p) {
                        fn.write_keys(pk);   // every warp's keys at its offset
                        SPEC_TRACE_EV(17, b, row, s, tot);
                    } else if (!bad && !oflow) {
                        // too many: the certified bound over every candidate, repeated
                        // until it stops rising (then it is the exact k-th value)
                        uint32_t o2, b2;
                        float vm2;
                        n = fn.finish(F, o2, b2, vm2);
                        uint64_t* list = sh.tk.cand;
                        for (int it = 0; it < 8 && n > A.cap_p; ++it) {
                            bool cert;
                            const uint32_t F2 = hist_bound_list(list, n, A.top_k, hkey(F), sh.hist, sh.scratch, cert);
                            if (!(cert && F2 > hkey(F))) break;
                            n = compact_list(list, n, F2, sh.ired);
                            F = static_cast<uint64_t>(F2) << 32;
                        }
                        if (n > A.cap_p) oflow = 1;   // ties at the k-th value: the fallback decides
                        else for (int i = threadIdx.x; i < n; i += kThreads) __stcg(pk + i, list[i]);
                        SPEC_TRACE_EV(17, b, row, s, tot | (1 << 20));
                    }
                    if (oflow || bad) n = 0;   // the combine does not read the keys then
                    if (threadIdx.x == 0) {
                        ph->flags = (bad ? kPfBad : 0u) | (oflow ? kPfOverflow : 0u) | (hint ? kPfHinted : 0u);
                        ph->cnt = n;
                        ph->kth = F;
                        ph->vmax = vm;
                        if (fn.dw.owns()) { ph->ly = wsl[0]; ph->qy = fn.dw.qy; }
                    }
                }
            } else {
                SumExpFn<E> fn;
                fn.c = A.c2;
                fn.dw = dw;
                ok = consume_row<E>(P, seq, plan, tma, x0, fn);
                if (ok) {
                    // per warp: fold (m_t, s_t) into the warp's max and sum; then thread 0
                    // folds the warps
                    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
                    float wm = fn.m;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
                    const float sc = (fn.s > 0.f) ? fn.s * ex2((fn.m - wm) * A.c2) : 0.f;
                    const dfloat ws = warp_sum_df(df_make(sc));
                    const uint32_t wb = __reduce_or_sync(0xffffffffu, fn.bad_flag());
                    if (lane == 0) { sh.wm[w] = wm; sh.ws[w] = make_float2(ws.hi, ws.lo); sh.wb[w] = wb; }
                    if (fn.dw.seen) wsl[0] = fn.dw.ly;
                    csync();
                    if (threadIdx.x == 0) {
                        float ms = -kInf;
                        uint32_t bad = 0;
                        for (int j = 0; j < kWarps; ++j) { ms = fmaxf(ms, sh.wm[j]); bad |= sh.wb[j]; }
                        dfloat tot = df_make(0.f);
                        for (int j = 0; j < kWarps; ++j)
                            if (sh.ws[j].x > 0.f) tot = df_add(tot, df_mul(ex2((sh.wm[j] - ms) * A.c2), df_of(sh.ws[j])));
                        ph->flags = bad ? kPfBad : 0u;
                        ph->cnt = 0;
                        ph->vmax = ms;
                        ph->sum = make_float2(tot.hi, tot.lo);
                        if (fn.dw.owns()) { ph->ly = wsl[0]; ph->qy = fn.dw.qy; }
                    }
                }
            }
        } else if (kind == kResid) {
            const ReqState* rs = &A.W.req[b];
            ResidFn<E> fn;
            fn.m = __ldcg(&rs->m);
            fn.c = A.c2;
            fn.invZ = __ldcg(&rs->invZ);
            ok = consume_row2<E>(P, seq, plan, tma, x0, fn);
            if (ok) {
                const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
                const dfloat wr = warp_sum_df(df_make(fn.r));
                const dfloat wp = warp_sum_df(df_make(fn.pw));
                if (lane == 0) { sh.ws[w] = make_float2(wr.hi, wr.lo); sh.ws2[w] = make_float2(wp.hi, wp.lo); }
                csync();
                if (threadIdx.x == 0) {
                    dfloat rsum = df_make(0.f), psum = df_make(0.f);
                    for (int j = 0; j < kWarps; ++j) { rsum = df_add(rsum, df_of(sh.ws[j])); psum = df_add(psum, df_of(sh.ws2[j])); }
                    ph->flags = 0;
                    ph->sum = make_float2(rsum.hi, rsum.lo);
                    ph->sum2 = make_float2(psum.hi, psum.lo);
                }
            }
        }
        if (!ok) break;
        SPEC_TRACE_EV(1, b, row, s, kind);
        csync();   // every consumer's partial writes are ordered before the hand-over
        Job j;
        j.task = t; j.slice = s; j.kind = kind; j.stop = 0; j.flags = 0;
        post_job(P, jseq, cseq, j, serve);
        SPEC_TRACE_EV(18, b, row, s, 0);
    }
    // stop the combiner once it has taken every job (serving its last combines)
    Job j;
    j.task.b = 0; j.task.row = 0; j.task.kind = 0; j.task.aux = 0; j.task.st = 0; j.task.base = 0;
    j.slice = 0; j.kind = 0; j.stop = 1; j.flags = 0;
    post_job(P, jseq, cseq, j, serve);
    // combines still in the combiner's queue are served until it stops
    consumer_wait(P, cseq, [&]() { return mbar_test(&P.jempty[(jseq - 1) % kJobs], ((jseq - 1) / kJobs) & 1u); }, serve);
}

// kCtasPerSm CTAs per SM (228 KiB of shared memory, 1 KiB reserved per CTA)
static_assert(kStages * kChunkBytes + sizeof(ChainSmem<true>) <= (228 * 1024) / kCtasPerSm - 1024,
              "chain CTA too large for kCtasPerSm per SM");

template <class E, bool kTopk>
static size_t chain_smem_bytes() {
    return kStages * kChunkBytes + sizeof(ChainSmem<kTopk>);
}

template <class E, bool kTopk>
static cudaError_t chain_launch(const ChainArgs& A, int grid, cudaStream_t st) {
    const size_t smem = chain_smem_bytes<E, kTopk>();
    cudaError_t e = cudaFuncSetAttribute(chain_kernel<E, kTopk>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    chain_kernel<E, kTopk><<<grid, kBlockThreads, smem, st>>>(A);
    return cudaGetLastError();
}

size_t chain_smem(int ldt, bool topk) {
    if (ldt == 0) return topk ? chain_smem_bytes<F32, true>() : chain_smem_bytes<F32, false>();
    return topk ? chain_smem_bytes<BF16, true>() : chain_smem_bytes<BF16, false>();
}

int chain_occupancy(int ldt, bool topk) {
    int n = 0;
    const int smem = static_cast<int>(chain_smem(ldt, topk));
    if (ldt == 0) {
        if (topk) { cudaFuncSetAttribute(chain_kernel<F32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_kernel<F32, true>, kBlockThreads, smem); }
        else { cudaFuncSetAttribute(chain_kernel<F32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
               cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_kernel<F32, false>, kBlockThreads, smem); }
    } else {
        if (topk) { cudaFuncSetAttribute(chain_kernel<BF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_kernel<BF16, true>, kBlockThreads, smem); }
        else { cudaFuncSetAttribute(chain_kernel<BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
               cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_kernel<BF16, false>, kBlockThreads, smem); }
    }
    return n;
}

cudaError_t chain_run(const ChainArgs& A, int grid, cudaStream_t st) {
    const bool topk = A.top_k > 0 && A.top_k < A.V;
    if (A.ldt == 0) return topk ? chain_launch<F32, true>(A, grid, st) : chain_launch<F32, false>(A, grid, st);
    return topk ? chain_launch<BF16, true>(A, grid, st) : chain_launch<BF16, false>(A, grid, st);
}

}  // namespace spec

SPEC_TRACE_EXPORT(chain)
