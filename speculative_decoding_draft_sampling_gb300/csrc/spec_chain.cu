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

// combine / slice-reduction scratch (the ring belongs to the producer):
// up to kScrKeys keys and as many ints
constexpr int kScrKeys = 2560;
template <bool kTopk> struct ChainTopkPart {};
template <> struct ChainTopkPart<true> {
    TopkSmem tk;
    alignas(16) unsigned char scr[kScrKeys * 12];
};

template <bool kTopk>
struct __align__(16) ChainSmem : ChainTopkPart<kTopk> {
    PipeSmem pipe;
    int last;
    int lcnt;
    int oflow;
    uint64_t sh64[4];
    double red[kWarps];
    int ired[kWarps + 4];
    int hist[64];
    uint32_t scratch[kWarps + 2];
    double dsh[8];
    int ish[8];
    float fsh[8];
    SliceHdrs hdrs;
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

// Commit the request: accepted drafts, then `last` (correction/bonus, or -1),
// then -1 padding.  All threads call; thread 0 publishes completion.
__device__ void chain_finish(const ChainArgs& A, int b, int n, int last, int st) {
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

// thread 0: push the request's next task after an accepted position
__device__ void chain_advance(const ChainArgs& A, int b, int row, int kb, int st, uint32_t hint) {
    ReqState* rs = &A.W.req[b];
    __stcg(&rs->status, st);
    Task t;
    t.b = b;
    t.row = row + 1;
    t.kind = (row + 1 < kb) ? kVerify : kBonus;
    t.aux = static_cast<int>(hint);
    push_task(A.W, t);
}

// acceptance of drafted y given p(y) and q(y): u < p/q (fp64)
__device__ __forceinline__ bool chain_accept(const ChainArgs& A, int y, double py, double qy, double u, int& st) {
    double ratio;
    if (y < 0 || y >= A.V) {
        st |= 8;
        ratio = 0.0;
    } else if (qy == 0.0) {
        st |= 2;
        ratio = py > 0.0 ? __longlong_as_double(0x7ff0000000000000LL) : 0.0;
    } else {
        ratio = py / qy;
    }
    return u < ratio;
}

// One warp: inverse CDF over n (token, weight) pairs sorted by token; the
// smallest token with prefix > t.  Result broadcast to the whole warp.
__device__ int warp_icdf_pairs(const int* tok, const double* w, int n, double t) {
    const int lane = threadIdx.x & 31;
    const int per = (n + 31) / 32;
    const int i0 = lane * per, i1 = min(n, i0 + per);
    double loc = 0.0;
    for (int i = i0; i < i1; ++i) loc += w[i];
    double inc = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
    }
    double c = inc - loc;
    int found = 0x7fffffff, lastpos = -1;
    for (int i = i0; i < i1; ++i) {
        if (w[i] > 0.0) {
            lastpos = i;
            c += w[i];
            if (c > t && found == 0x7fffffff) found = i;
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

__device__ __forceinline__ int n_slices_dbg(int S) { return S; }

// Filter hint for the next row from this row's top-k threshold tau and max
// m: half the gap below tau (rows of one target differ little in tau).
__device__ __forceinline__ uint32_t next_hint(float tau, float m) {
    const float h = tau - 0.5f * (m - tau);
    return (h == h && h > -kInf) ? fkey(h) : 0u;
}

// ---------------------------------------------------------------------------
// combine with top-k: the candidate lists of all slices hold S exactly
// ---------------------------------------------------------------------------
template <class E>
__device__ void chain_fallback(const ChainArgs& A, ChainSmem<true>& sh, int b, int row, int kind,
                               int st, float vmax);

template <class E>
__device__ void combine_topk(const ChainArgs& A, ChainSmem<true>& sh, int b, int row,
                             int kind, int st) {
    const int S = A.S;
    const int k = A.top_k;
    const int kb = chain_k(A, b);
    // independent loads first: they overlap the header loads
    const double uk = static_cast<double>(chain_u(A, b, kb));
    const double ur = kind == kVerify ? static_cast<double>(chain_u(A, b, row)) : 0.0;
    const int y = kind == kVerify ? A.draft[static_cast<long long>(b) * A.K + row] : -1;
    SliceHdrs& H = sh.hdrs;
    load_hdrs(A.W, b, S, H);
    SPEC_TRACE_EV(5, b, row, n_slices_dbg(S), kind);
    uint32_t flags = 0;
    float vmax = -kInf;
    uint64_t theta = 0;
    for (int s = 0; s < S; ++s) {
        flags |= H.flags[s];
        vmax = max_nan(vmax, H.vmax[s]);
        theta = H.kth[s] > theta ? H.kth[s] : theta;
    }
    if ((flags & kPfBad) || !(vmax > -kInf)) {
        chain_finish(A, b, row, -1, st | 1);
        return;
    }
    if (flags & kPfOverflow) {
        chain_fallback<E>(A, sh, b, row, kind, st, vmax);
        return;
    }
    const bool hinted = (flags & kPfHinted) != 0;
    // gather every candidate at or above the largest slice filter
    constexpr int kList = kScrKeys;
    uint64_t* list = reinterpret_cast<uint64_t*>(sh.scr);
    int* rank = reinterpret_cast<int*>(sh.scr + kList * 8);
    gather_keys(A.W, b, S, H, [&](uint64_t key) { return key >= theta; }, list, kList, &sh.lcnt, &sh.oflow);
    int n = sh.lcnt;
    SPEC_TRACE_EV(6, b, row, n, kind);
    if (sh.oflow || n > kList) {
        csync();
        chain_fallback<E>(A, sh, b, row, kind, st, vmax);
        return;
    }
    if (n < k) {
        csync();
        if (hinted) {
            // the hint was above the row's k-th value: stream the row again without it
            if (threadIdx.x == 0) {
                __stcg(&A.W.req[b].status, st);
                Task t;
                t.b = b; t.row = row; t.kind = kind | kNoHint; t.aux = 0;
                push_task(A.W, t);
            }
            return;
        }
        chain_fallback<E>(A, sh, b, row, kind, st, vmax);
        return;
    }
    if (n > 2 * k + 64) {
        // certified pre-reduction: fewer keys for the quadratic selection
        bool cert;
        const uint32_t F = hist_bound_list(list, n, k, hkey(theta), sh.hist, sh.scratch, cert);
        if (cert && F > hkey(theta)) n = compact_list(list, n, F, sh.ired);
    }
    uint64_t kth;
    bool of = false;
    uint64_t* cand = sh.tk.cand;
    constexpr int kCandCap = kWarps * TopkSmem::kRegion;
    const int keep = select_to(list, n, k, true, rank, cand, kCandCap, kth, of, sh.sh64, sh.ired);
    SPEC_TRACE_EV(7, b, row, n, kind);
    if (of) {
        chain_fallback<E>(A, sh, b, row, kind, st, vmax);
        return;
    }
    // S = cand[0 .. keep): values >= tau, sorted by value descending
    const uint32_t tau_key = hkey(cand[keep - 1]);
    const float tau = ckey_val(cand[keep - 1]);
    const float m = vmax, c2 = A.c2;
    double zpart = 0.0;
    for (int i = threadIdx.x; i < keep; i += kThreads)
        zpart += static_cast<double>(ex2((ckey_val(cand[i]) - m) * c2));
    const double Z = block_sum_d(zpart, sh.red);
    const uint32_t hint = next_hint(tau, m);
    if (threadIdx.x == 0) __stcg(&A.W.ctrl->hint0, hint);

    // weights of S sorted by token id (ascending): pairs in the ring
    int* tok = reinterpret_cast<int*>(sh.scr);
    double* wgt = reinterpret_cast<double*>(sh.scr + kScrKeys * 4);
    auto sort_by_token = [&](bool residual, const float* qrow, double& total) {
        double part = 0.0;
        for (int i = threadIdx.x; i < keep; i += kThreads) {
            const int x = ckey_idx(cand[i]);
            int r = 0;
            for (int j = 0; j < keep; ++j) r += ckey_idx(cand[j]) < x;
            const double p = static_cast<double>(ex2((ckey_val(cand[i]) - m) * c2)) / Z;
            double w = p;
            if (residual) {
                const float qx = (x >= 0 && x < A.V) ? qrow[x] : 0.f;   // keys always hold in-range ids
                const double d = p - static_cast<double>(qx);
                w = d > 0.0 ? d : 0.0;
            }
            tok[r] = x;
            wgt[r] = w;
            part += w;
        }
        total = block_sum_d(part, sh.red);
    };

    if (kind == kVerify) {
        double py = 0.0, qy = 0.0;
        if (y >= 0 && y < A.V) {
            const int sy = y / A.SL;
            const float ly = H.ly[sy];
            qy = static_cast<double>(H.qy[sy]);
            if (fkey(ly) >= tau_key) py = static_cast<double>(ex2((ly - m) * c2)) / Z;
        }
        const bool acc = chain_accept(A, y, py, qy, ur, st);
        if (acc) {
            if (threadIdx.x == 0) {
                chain_diag(A, b, row, (float)py, (float)qy, (float)Z, 0.f);
                chain_advance(A, b, row, kb, st, hint);
            }
            return;
        }
        // residual [p - q]_+ lives on S (p = 0 outside it)
        double R_mass;
        sort_by_token(true, chain_qrow(A, b, row), R_mass);
        if (!(R_mass > 0.0)) {
            st |= 4;
            sort_by_token(false, nullptr, R_mass);
        }
        int x = -1;
        if (threadIdx.x < 32) x = warp_icdf_pairs(tok, wgt, keep, uk * R_mass);
        if (threadIdx.x == 0) {
            sh.ish[0] = x;
            chain_diag(A, b, row, (float)py, (float)qy, (float)Z, (st & 4) ? 0.f : (float)R_mass);
        }
        csync();
        chain_finish(A, b, row, sh.ish[0], st);
        return;
    }
    // bonus row: draw from p
    double tot;
    sort_by_token(false, nullptr, tot);
    int x = -1;
    if (threadIdx.x < 32) x = warp_icdf_pairs(tok, wgt, keep, uk * tot);
    if (threadIdx.x == 0) sh.ish[0] = x;
    csync();
    x = sh.ish[0];
    if (threadIdx.x == 0 && x >= 0 && x < A.V)
        chain_diag(A, b, row, (float)(static_cast<double>(ex2((E::load(chain_lrow<E>(A, b, row), x) - m) * c2)) / Z),
                   0.f, (float)Z, 0.f);
    chain_finish(A, b, row, x, st);
}

// Exact single-CTA path for rows whose top-k set did not fit the candidate
// buffers (massive ties, adversarial order): tau by bisection over
// order-preserving keys, then full-row passes.  Slow; correctness only.
template <class E>
__device__ void chain_fallback(const ChainArgs& A, ChainSmem<true>& sh, int b, int row, int kind,
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
    const double Z = cta_sum(0, V, wp, sh.red);
    const int kb = chain_k(A, b);
    const double uk = static_cast<double>(chain_u(A, b, kb));
    if (kind == kVerify) {
        const int y = A.draft[static_cast<long long>(b) * A.K + row];
        double py = 0.0, qy = 0.0;
        if (y >= 0 && y < V) {
            py = static_cast<double>(wp(y)) / Z;
            qy = static_cast<double>(chain_qrow(A, b, row)[y]);
        }
        if (chain_accept(A, y, py, qy, static_cast<double>(chain_u(A, b, row)), st)) {
            if (threadIdx.x == 0) {
                chain_diag(A, b, row, (float)py, (float)qy, (float)Z, 0.f);
                chain_advance(A, b, row, kb, st, 0u);
            }
            return;
        }
        const float* qrow = chain_qrow(A, b, row);
        const float invZ = static_cast<float>(1.0 / Z);
        auto wr = [&](int x) -> float {
            const float d = wp(x) * invZ - qrow[x];
            return d > 0.f ? d : 0.f;
        };
        const double R_mass = cta_sum(0, V, wr, sh.red);
        int x;
        if (R_mass > 0.0) {
            x = cta_icdf(0, V, uk * R_mass, wr, sh.red, sh.ired);
        } else {
            st |= 4;
            x = cta_icdf(0, V, uk * Z, wp, sh.red, sh.ired);
        }
        if (threadIdx.x == 0) chain_diag(A, b, row, (float)py, (float)qy, (float)Z, (float)R_mass);
        chain_finish(A, b, row, x, st);
        return;
    }
    const int x = cta_icdf(0, V, uk * Z, wp, sh.red, sh.ired);
    if (threadIdx.x == 0)
        chain_diag(A, b, row, (float)(static_cast<double>(wp(x)) / Z), 0.f, (float)Z, 0.f);
    chain_finish(A, b, row, x, st);
}

// ---------------------------------------------------------------------------
// combine without truncation: per-slice (max, sum of 2^((l-m_s)c))
// ---------------------------------------------------------------------------
// index of the slice whose running prefix of `val(s)` crosses t; *before* =
// prefix before it.  Thread 0 computes, result broadcast.
template <class F>
__device__ int find_slice(int S, double t, F val, double& before, double* dsh, int* ish) {
    if (threadIdx.x == 0) {
        double acc = 0.0;
        int pick = -1, lastpos = -1;
        double lastbefore = 0.0;
        for (int s = 0; s < S; ++s) {
            const double v = val(s);
            if (v > 0.0) {
                if (acc + v > t) { pick = s; break; }
                lastpos = s;
                lastbefore = acc;
            }
            acc += v;
        }
        if (pick < 0) { pick = lastpos >= 0 ? lastpos : 0; acc = lastbefore; }
        ish[0] = pick;
        dsh[0] = acc;
    }
    csync();
    const int s = ish[0];
    before = dsh[0];
    csync();
    return s;
}

template <class E>
__device__ void combine_full(const ChainArgs& A, ChainSmem<false>& sh, int b, int row, int kind, int st) {
    const int S = A.S;
    const int kb = chain_k(A, b);
    const double cd = static_cast<double>(A.c2);
    const double uk = static_cast<double>(chain_u(A, b, kb));
    const double ur = kind == kVerify ? static_cast<double>(chain_u(A, b, row)) : 0.0;
    const int y = kind == kVerify ? A.draft[static_cast<long long>(b) * A.K + row] : -1;
    const void* lrow = chain_lrow<E>(A, b, row);
    SliceHdrs& H = sh.hdrs;
    load_hdrs(A.W, b, S, H);
    SPEC_TRACE_EV(5, b, row, S, kind);
    if (kind == kResid) {
        const ReqState* rs = &A.W.req[b];
        const float m = static_cast<float>(__ldcg(&rs->m));
        const double Z = __ldcg(&rs->Z);
        double R_mass = 0.0, P_mass = 0.0;
        for (int s = 0; s < S; ++s) {
            R_mass += H.sum[s];
            P_mass += H.sum2[s];
        }
        const float* qrow = chain_qrow(A, b, row);
        const float c2 = A.c2, invZ = static_cast<float>(1.0 / Z);
        int x;
        double before;
        if (R_mass > 0.0) {
            const double t = uk * R_mass;
            const int s = find_slice(S, t, [&](int j) { return H.sum[j]; }, before, sh.dsh, sh.ish);
            auto wr = [&](int xx) -> float {
                const float d = ex2((E::load(lrow, xx) - m) * c2) * invZ - qrow[xx];
                return d > 0.f ? d : 0.f;
            };
            const int x0 = s * A.SL, x1 = min(A.V, x0 + A.SL);
            x = cta_icdf(x0, x1, t - before, wr, sh.red, sh.ired);
        } else {
            st |= 4;
            const double t = uk * P_mass;
            const int s = find_slice(S, t, [&](int j) { return H.sum2[j]; }, before, sh.dsh, sh.ish);
            auto wp = [&](int xx) -> float { return ex2((E::load(lrow, xx) - m) * c2); };
            const int x0 = s * A.SL, x1 = min(A.V, x0 + A.SL);
            x = cta_icdf(x0, x1, t - before, wp, sh.red, sh.ired);
        }
        if (threadIdx.x == 0 && A.diag)
            A.diag[(static_cast<long long>(b) * (A.K + 1) + row) * 4 + 3] = (st & 4) ? 0.f : (float)R_mass;
        chain_finish(A, b, row, x, st);
        return;
    }
    // VERIFY or BONUS: max and normaliser from the slice partials
    uint32_t flags = 0;
    float vmax = -kInf;
    for (int s = 0; s < S; ++s) {
        flags |= H.flags[s];
        vmax = max_nan(vmax, H.vmax[s]);
    }
    if ((flags & kPfBad) || !(vmax > -kInf)) {
        chain_finish(A, b, row, -1, st | 1);
        return;
    }
    const double m = static_cast<double>(vmax);
    auto scaled = [&](int s) -> double {
        const double sm = H.sum[s];
        return sm > 0.0 ? sm * exp2((static_cast<double>(H.vmax[s]) - m) * cd) : 0.0;
    };
    double zp = 0.0;
    for (int s = threadIdx.x; s < S; s += kThreads) zp += scaled(s);
    const double Z = block_sum_d(zp, sh.red);
    SPEC_TRACE_EV(6, b, row, S, kind);
    if (kind == kVerify) {
        double py = 0.0, qy = 0.0;
        if (y >= 0 && y < A.V) {
            const int sy = y / A.SL;
            py = exp((static_cast<double>(H.ly[sy]) - m) / A.Td) / Z;
            qy = static_cast<double>(H.qy[sy]);
        }
        const bool acc = chain_accept(A, y, py, qy, ur, st);
        SPEC_TRACE_EV(7, b, row, S, kind);
        if (threadIdx.x == 0) chain_diag(A, b, row, (float)py, (float)qy, (float)Z, 0.f);
        if (acc) {
            if (threadIdx.x == 0) chain_advance(A, b, row, kb, st, 0u);
            return;
        }
        if (threadIdx.x == 0) {
            ReqState* rs = &A.W.req[b];
            __stcg(&rs->m, m);
            __stcg(&rs->Z, Z);
            __stcg(&rs->status, st);
            Task t;
            t.b = b; t.row = row; t.kind = kResid; t.aux = 0;
            push_task(A.W, t);
        }
        return;
    }
    // BONUS: inverse CDF of p; find the slice, then rescan it
    const double t = uk * Z;
    double before;
    const int s = find_slice(S, t, scaled, before, sh.dsh, sh.ish);
    const float mf = vmax, c2 = A.c2;
    auto wp = [&](int xx) -> float { return ex2((E::load(lrow, xx) - mf) * c2); };
    const int x0 = s * A.SL, x1 = min(A.V, x0 + A.SL);
    const int x = cta_icdf(x0, x1, t - before, wp, sh.red, sh.ired);
    if (threadIdx.x == 0)
        chain_diag(A, b, row, (float)(exp((static_cast<double>(E::load(lrow, x)) - m) / A.Td) / Z), 0.f,
                   (float)Z, 0.f);
    chain_finish(A, b, row, x, st);
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
    const int x0 = slice * A.SL, x1 = min(A.V, x0 + A.SL);
    if (kind == kVerify || kind == kBonus) return plan_single(chain_lrow<E>(A, t.b, t.row), E::kBytes, x0, x1);
    if (kind == kResid) return plan_dual(chain_lrow<E>(A, t.b, t.row), E::kBytes, chain_qrow(A, t.b, t.row), x0, x1);
    return plan_none();
}

template <class E, bool kTopk>
__global__ void __launch_bounds__(kBlockThreads, 2) chain_kernel(const ChainArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    auto& sh = *reinterpret_cast<ChainSmem<kTopk>*>(smem + kStages * kChunkBytes);
    const Pipe P = pipe_init(smem, sh.pipe);
    // the residual pass streams q beside the logits; without q rows (K = 0)
    // there is no residual pass
    const bool tma = A.tma_l && (kTopk || A.K == 0 || A.tma_q);
    if (threadIdx.x >= kThreads) {
        if (threadIdx.x == kThreads) {
            producer_loop(A.W, A.B, A.S, P, tma,
                          [&](Claimed& c) {
                              if (kTopk && c.task.kind < 0) c.hint = __ldcg(&A.W.ctrl->hint0);
                          },
                          [&](const Claimed& c) {
                              return chain_plan<E>(A, c.task, chain_unit_kind<E>(A, c.task), c.slice);
                          });
        }
        return;
    }
    uint32_t seq = 0;
    for (uint32_t u = 0;; ++u) {
        const Claimed cl = next_unit(P, u);
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
        const int x0 = s * A.SL, x1 = min(A.V, x0 + A.SL);
        const StreamPlan plan = chain_plan<E>(A, t, kind, s);
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
                fn.init(&sh.tk, A.top_k, hint);
                fn.dw = dw;
                if (!consume_row<E>(P, seq, plan, tma, x0, fn)) break;
                SPEC_TRACE_EV(4, b, row, s, kind);
                uint64_t F;
                uint32_t oflow, bad;
                int n = fn.finish(F, oflow, bad);
                uint64_t* list = sh.tk.cand;
                const float vm = block_max_nan(fn.vmx, reinterpret_cast<float*>(sh.red));
                if (fn.dw.seen) wsl[0] = fn.dw.ly;
                if (n > A.cap_p && !oflow && !bad) {
                    // certified bound first, then the exact top-k (ties kept)
                    bool cert;
                    const uint32_t F2 = hist_bound_list(list, n, A.top_k, hkey(F), sh.hist, sh.scratch, cert);
                    if (cert && F2 > hkey(F)) {
                        n = compact_list(list, n, F2, sh.ired);
                        F = static_cast<uint64_t>(F2) << 32;
                    }
                    if (n > A.cap_p) {
                        uint64_t* dst = reinterpret_cast<uint64_t*>(sh.scr);
                        int* rank = reinterpret_cast<int*>(sh.scr + kScrKeys * 8);
                        uint64_t kth;
                        bool of2;
                        const int keep = select_to(list, n, A.top_k, true, rank, dst, min(A.cap_p, kScrKeys), kth,
                                                   of2, sh.sh64, sh.ired);
                        if (of2) oflow = 1;
                        else F = static_cast<uint64_t>(hkey(kth)) << 32;
                        n = keep;
                        list = dst;
                    }
                }
                if (oflow || bad) n = 0;   // the combine does not read the keys then
                csync();
                for (int i = threadIdx.x; i < n; i += kThreads) __stcg(pk + i, list[i]);
                if (threadIdx.x == 0) {
                    ph->flags = (bad ? kPfBad : 0u) | (oflow ? kPfOverflow : 0u) | (hint ? kPfHinted : 0u);
                    ph->cnt = n;
                    ph->kth = F;
                    ph->vmax = vm;
                    if (fn.dw.owns()) { ph->ly = wsl[0]; ph->qy = fn.dw.qy; }
                }
            } else {
                SumExpFn<E> fn;
                fn.c = A.c2;
                fn.dw = dw;
                if (!consume_row<E>(P, seq, plan, tma, x0, fn)) break;
                // fold per-thread (m_t, s_t) into the slice max and sum
                const uint64_t mk = block_max_u64(static_cast<uint64_t>(fkey(fn.m)), reinterpret_cast<uint64_t*>(sh.red));
                const float ms = fkey_inv(static_cast<uint32_t>(mk));
                float sc = 0.f;
                if (fn.s > 0.f) sc = fn.s * ex2((fn.m - ms) * A.c2);
                const double tot = block_sum_d(static_cast<double>(sc), sh.red);
                const uint32_t bad = block_or(fn.bad_flag(), reinterpret_cast<uint32_t*>(sh.red));
                if (fn.dw.seen) wsl[0] = fn.dw.ly;
                csync();
                if (threadIdx.x == 0) {
                    ph->flags = bad ? kPfBad : 0u;
                    ph->cnt = 0;
                    ph->vmax = ms;
                    ph->sum = tot;
                    if (fn.dw.owns()) { ph->ly = wsl[0]; ph->qy = fn.dw.qy; }
                }
            }
        } else if (kind == kResid) {
            const ReqState* rs = &A.W.req[b];
            ResidFn<E> fn;
            fn.m = static_cast<float>(__ldcg(&rs->m));
            fn.c = A.c2;
            fn.invZ = static_cast<float>(1.0 / __ldcg(&rs->Z));
            if (!consume_row2<E>(P, seq, plan, tma, x0, fn)) break;
            const double rsum = block_sum_d(static_cast<double>(fn.r), sh.red);
            const double psum = block_sum_d(static_cast<double>(fn.pw), sh.red);
            if (threadIdx.x == 0) {
                ph->flags = 0;
                ph->sum = rsum;
                ph->sum2 = psum;
            }
        }
        SPEC_TRACE_EV(1, b, row, s, kind);
        if (arrive(A.W, b, A.S, &sh.last)) {
            SPEC_TRACE_EV(2, b, row, s, kind);
            const int st = initial ? 0 : __ldcg(&A.W.req[b].status);
            if (kind == kInvalid) {
                chain_finish(A, b, 0, -1, 16);
            } else if constexpr (kTopk) {
                combine_topk<E>(A, sh, b, row, kind, st);
            } else {
                combine_full<E>(A, sh, b, row, kind, st);
            }
            csync();
            SPEC_TRACE_EV(3, b, row, s, kind);
        }
    }
}

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
