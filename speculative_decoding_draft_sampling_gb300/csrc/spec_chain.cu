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

template <int kCap>
struct __align__(16) ChainSmem {
    uint64_t bars[kStages];
    Claimed claimed;
    int last;
    int cnt;
    int oflow;
    int lcnt;
    uint64_t sh64[4];
    double red[kWarps];
    int ired[kWarps + 4];
    uint64_t pool[kThreads];
    double dsh[8];
    int ish[8];
    uint64_t cand[kCap];
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
    __syncthreads();
    if (threadIdx.x == 0) finish_request(A.W);
}

__device__ __forceinline__ void chain_diag(const ChainArgs& A, int b, int i, float py, float qy, float Z, float R) {
    if (!A.diag) return;
    float* d = A.diag + (static_cast<long long>(b) * (A.K + 1) + i) * 4;
    d[0] = py; d[1] = qy; d[2] = Z; d[3] = R;
}

// push the request's next task after an accepted position
__device__ void chain_advance(const ChainArgs& A, int b, int row, int kb, int st) {
    if (threadIdx.x == 0) {
        ReqState* rs = &A.W.req[b];
        __stcg(&rs->status, st);
        Task t;
        t.b = b;
        t.row = row + 1;
        t.kind = (row + 1 < kb) ? kVerify : kBonus;
        t.aux = 0;
        push_task(A.W, t);
    }
}

// acceptance of drafted y at one row, given p(y) (fp64): returns accept
__device__ bool chain_accept(const ChainArgs& A, int b, int row, int y, double py, double& qy, int& st) {
    double ratio;
    if (y < 0 || y >= A.V) {
        st |= 8;
        qy = 0.0;
        ratio = 0.0;
    } else {
        qy = static_cast<double>(chain_qrow(A, b, row)[y]);
        if (qy == 0.0) {
            st |= 2;
            ratio = py > 0.0 ? __longlong_as_double(0x7ff0000000000000LL) : 0.0;
        } else {
            ratio = py / qy;
        }
    }
    const double u = static_cast<double>(A.uniforms[static_cast<long long>(b) * (A.K + 1) + row]);
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

// ---------------------------------------------------------------------------
// combine with top-k: the candidate lists of all slices hold S exactly
// ---------------------------------------------------------------------------
template <class E, int kCap>
__device__ void combine_topk(const ChainArgs& A, Ring& R, ChainSmem<kCap>& sh, int b, int row,
                             int kind, int st);

template <class E, int kCap>
__device__ void chain_fallback(const ChainArgs& A, ChainSmem<kCap>& sh, int b, int row, int kind,
                               int st, float vmax);

template <class E, int kCap>
__device__ void combine_topk(const ChainArgs& A, Ring& R, ChainSmem<kCap>& sh, int b, int row,
                             int kind, int st) {
    const int S = A.S;
    const int k = A.top_k;
    uint32_t flags = 0;
    uint64_t vkey = 0, theta = 0;
    for (int s = threadIdx.x; s < S; s += kThreads) {
        const PartHdr* h = part_hdr(A.W, b, s, S);
        flags |= __ldcg(&h->flags);
        const int c = __ldcg(&h->cnt);
        if (c > 0) {
            const uint64_t k0 = __ldcg(part_keys(A.W, b, s, S));
            vkey = k0 > vkey ? k0 : vkey;
        }
        const uint64_t kk = __ldcg(&h->kth);
        if (c >= k) theta = kk > theta ? kk : theta;
    }
    flags = block_or(flags, reinterpret_cast<uint32_t*>(sh.red));
    vkey = block_max_u64(vkey, reinterpret_cast<uint64_t*>(sh.red));
    theta = block_max_u64(theta, reinterpret_cast<uint64_t*>(sh.red));
    const float vmax = vkey ? ckey_val(vkey) : -kInf;
    const int kb = chain_k(A, b);
    if ((flags & kPfBad) || !(vmax > -kInf)) {
        chain_finish(A, b, row, -1, st | 1);
        return;
    }
    if (flags & kPfOverflow) {
        chain_fallback<E, kCap>(A, sh, b, row, kind, st, vmax);
        return;
    }
    // gather every candidate whose value reaches the largest slice threshold
    constexpr int kList = 4096;                      // keys in the ring (32 KiB)
    uint64_t* list = reinterpret_cast<uint64_t*>(R.buf);
    int* rank = reinterpret_cast<int*>(R.buf + kList * 8);
    const uint32_t th = static_cast<uint32_t>(theta >> 32);
    if (threadIdx.x == 0) { sh.lcnt = 0; sh.oflow = 0; }
    __syncthreads();
    for (int s = 0; s < S; ++s) {
        const int c = __ldcg(&part_hdr(A.W, b, s, S)->cnt);
        const uint64_t* keys = part_keys(A.W, b, s, S);
        for (int i0 = 0; i0 < c; i0 += kThreads) {
            const int i = i0 + threadIdx.x;
            uint64_t key = 0;
            bool p = false;
            if (i < c) {
                key = __ldcg(keys + i);
                p = static_cast<uint32_t>(key >> 32) >= th;
            }
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            int base = 0;
            const int lane = threadIdx.x & 31;
            if (lane == 0 && bal) base = atomicAdd(&sh.lcnt, __popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (p) {
                const int pos = base + __popc(bal & ((1u << lane) - 1u));
                if (pos < kList) list[pos] = key;
                else sh.oflow = 1;
            }
        }
    }
    __syncthreads();
    int n = sh.lcnt;
    if (sh.oflow || n > kList) {
        __syncthreads();
        chain_fallback<E, kCap>(A, sh, b, row, kind, st, vmax);
        return;
    }
    uint64_t kth;
    bool of = false;
    const int keep = select_to(list, n, k, true, rank, sh.cand, kCap, kth, of, sh.sh64, sh.ired);
    if (of) {
        chain_fallback<E, kCap>(A, sh, b, row, kind, st, vmax);
        return;
    }
    // S = sh.cand[0 .. keep): values >= tau, sorted by value descending
    const uint32_t tau_key = static_cast<uint32_t>(sh.cand[keep - 1] >> 32);
    const double m = static_cast<double>(vmax);
    const double T = A.Td;
    double zpart = 0.0;
    for (int i = threadIdx.x; i < keep; i += kThreads)
        zpart += exp((static_cast<double>(ckey_val(sh.cand[i])) - m) / T);
    const double Z = block_sum_d(zpart, sh.red);
    const double uk = static_cast<double>(A.uniforms[static_cast<long long>(b) * (A.K + 1) + kb]);

    // weights of S sorted by token id (ascending): pairs in the ring
    int* tok = reinterpret_cast<int*>(R.buf);
    double* wgt = reinterpret_cast<double*>(R.buf + 16384);
    auto sort_by_token = [&](bool residual, const float* qrow, double& total) {
        double part = 0.0;
        for (int i = threadIdx.x; i < keep; i += kThreads) {
            const int x = ckey_idx(sh.cand[i]);
            int r = 0;
            for (int j = 0; j < keep; ++j) r += ckey_idx(sh.cand[j]) < x;
            const double p = exp((static_cast<double>(ckey_val(sh.cand[i])) - m) / T) / Z;
            double w = p;
            if (residual) {
                const double d = p - static_cast<double>(qrow[x]);
                w = d > 0.0 ? d : 0.0;
            }
            tok[r] = x;
            wgt[r] = w;
            part += w;
        }
        total = block_sum_d(part, sh.red);
    };

    if (kind == kVerify) {
        const int y = A.draft[static_cast<long long>(b) * A.K + row];
        double py = 0.0;
        if (y >= 0 && y < A.V) {
            const float vy = E::load(chain_lrow<E>(A, b, row), y);
            if (fkey(vy) >= tau_key) py = exp((static_cast<double>(vy) - m) / T) / Z;
        }
        double qy;
        const bool acc = chain_accept(A, b, row, y, py, qy, st);
        if (acc) {
            if (threadIdx.x == 0) chain_diag(A, b, row, (float)py, (float)qy, (float)Z, 0.f);
            chain_advance(A, b, row, kb, st);
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
        __syncthreads();
        chain_finish(A, b, row, sh.ish[0], st);
        return;
    }
    // bonus row: draw from p
    double tot;
    sort_by_token(false, nullptr, tot);
    int x = -1;
    if (threadIdx.x < 32) x = warp_icdf_pairs(tok, wgt, keep, uk * tot);
    if (threadIdx.x == 0) sh.ish[0] = x;
    __syncthreads();
    x = sh.ish[0];
    if (threadIdx.x == 0 && x >= 0)
        chain_diag(A, b, row, (float)(exp((static_cast<double>(E::load(chain_lrow<E>(A, b, row), x)) - m) / T) / Z),
                   0.f, (float)Z, 0.f);
    chain_finish(A, b, row, x, st);
}

// Exact single-CTA path for rows whose top-k set did not fit the candidate
// buffers (massive ties): tau by bisection over order-preserving keys, then
// full-row passes.  Slow; correctness only.
template <class E, int kCap>
__device__ void chain_fallback(const ChainArgs& A, ChainSmem<kCap>& sh, int b, int row, int kind,
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
    const double uk = static_cast<double>(A.uniforms[static_cast<long long>(b) * (A.K + 1) + kb]);
    if (kind == kVerify) {
        const int y = A.draft[static_cast<long long>(b) * A.K + row];
        double py = 0.0;
        if (y >= 0 && y < V) {
            const float vy = E::load(lrow, y);
            if (fkey(vy) >= tau) py = exp((static_cast<double>(vy) - m) / A.Td) / Z;
        }
        double qy;
        if (chain_accept(A, b, row, y, py, qy, st)) {
            if (threadIdx.x == 0) chain_diag(A, b, row, (float)py, (float)qy, (float)Z, 0.f);
            chain_advance(A, b, row, kb, st);
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
    __syncthreads();
    const int s = ish[0];
    before = dsh[0];
    __syncthreads();
    return s;
}

template <class E, int kCap>
__device__ void combine_full(const ChainArgs& A, ChainSmem<kCap>& sh, int b, int row, int kind, int st) {
    const int S = A.S;
    const int kb = chain_k(A, b);
    const double cd = static_cast<double>(A.c2);
    const double uk = static_cast<double>(A.uniforms[static_cast<long long>(b) * (A.K + 1) + kb]);
    const void* lrow = chain_lrow<E>(A, b, row);
    if (kind == kResid) {
        const ReqState* rs = &A.W.req[b];
        const float m = static_cast<float>(__ldcg(&rs->m));
        const double Z = __ldcg(&rs->Z);
        double rp = 0.0, pp = 0.0;
        for (int s = threadIdx.x; s < S; s += kThreads) {
            const PartHdr* h = part_hdr(A.W, b, s, S);
            rp += __ldcg(&h->sum);
            pp += __ldcg(&h->sum2);
        }
        const double R_mass = block_sum_d(rp, sh.red);
        const double P_mass = block_sum_d(pp, sh.red);
        const float* qrow = chain_qrow(A, b, row);
        const float c2 = A.c2, invZ = static_cast<float>(1.0 / Z);
        int x;
        double before;
        if (R_mass > 0.0) {
            const double t = uk * R_mass;
            const int s = find_slice(S, t, [&](int j) { return __ldcg(&part_hdr(A.W, b, j, S)->sum); },
                                     before, sh.dsh, sh.ish);
            auto wr = [&](int xx) -> float {
                const float d = ex2((E::load(lrow, xx) - m) * c2) * invZ - qrow[xx];
                return d > 0.f ? d : 0.f;
            };
            const int x0 = s * A.SL, x1 = min(A.V, x0 + A.SL);
            x = cta_icdf(x0, x1, t - before, wr, sh.red, sh.ired);
        } else {
            st |= 4;
            const double t = uk * P_mass;
            const int s = find_slice(S, t, [&](int j) { return __ldcg(&part_hdr(A.W, b, j, S)->sum2); },
                                     before, sh.dsh, sh.ish);
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
    float vm = -kInf;
    for (int s = threadIdx.x; s < S; s += kThreads) {
        const PartHdr* h = part_hdr(A.W, b, s, S);
        flags |= __ldcg(&h->flags);
        vm = fmaxf(vm, __ldcg(&h->vmax));
    }
    flags = block_or(flags, reinterpret_cast<uint32_t*>(sh.red));
    const uint64_t vk = block_max_u64(static_cast<uint64_t>(fkey(vm)), reinterpret_cast<uint64_t*>(sh.red));
    const float vmax = fkey_inv(static_cast<uint32_t>(vk));
    if ((flags & kPfBad) || !(vmax > -kInf)) {
        chain_finish(A, b, row, -1, st | 1);
        return;
    }
    const double m = static_cast<double>(vmax);
    auto scaled = [&](int s) -> double {
        const PartHdr* h = part_hdr(A.W, b, s, S);
        const double ms = static_cast<double>(__ldcg(&h->vmax));
        const double sm = __ldcg(&h->sum);
        return sm > 0.0 ? sm * exp2((ms - m) * cd) : 0.0;
    };
    double zp = 0.0;
    for (int s = threadIdx.x; s < S; s += kThreads) zp += scaled(s);
    const double Z = block_sum_d(zp, sh.red);
    if (kind == kVerify) {
        const int y = A.draft[static_cast<long long>(b) * A.K + row];
        double py = 0.0;
        if (y >= 0 && y < A.V) py = exp((static_cast<double>(E::load(lrow, y)) - m) / A.Td) / Z;
        double qy;
        const bool acc = chain_accept(A, b, row, y, py, qy, st);
        if (threadIdx.x == 0) chain_diag(A, b, row, (float)py, (float)qy, (float)Z, 0.f);
        if (acc) {
            chain_advance(A, b, row, kb, st);
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
template <class E, bool kTopk>
__global__ void __launch_bounds__(kThreads) chain_kernel(const ChainArgs A) {
    constexpr int kCap = kThreads * E::kVec + 512;
    extern __shared__ __align__(128) unsigned char smem[];
    auto& sh = *reinterpret_cast<ChainSmem<kCap>*>(smem + kStages * kChunkBytes);
    Ring R;
    R.init(smem, sh.bars);
    for (;;) {
        Task t;
        int s;
        if (!claim(A.W, A.B, A.S, t, s, &sh.claimed)) break;
        const int b = t.b;
        int kind = t.kind, row = t.row;
        const bool initial = kind < 0;
        if (initial) {
            const int kb = chain_k(A, b);
            kind = (kb < 0 || kb > A.K) ? kInvalid : (kb == 0 ? kBonus : kVerify);
        }
        PartHdr* ph = part_hdr(A.W, b, s, A.S);
        uint64_t* pk = part_keys(A.W, b, s, A.S);
        const int x0 = s * A.SL, x1 = min(A.V, x0 + A.SL);
        if (kind == kVerify || kind == kBonus) {
            const void* lrow = chain_lrow<E>(A, b, row);
            if constexpr (kTopk) {
                if (threadIdx.x == 0) { sh.cnt = 0; sh.oflow = 0; }
                __syncthreads();
                TopkFn<E, true, kCap> fn;
                fn.cand = sh.cand; fn.cnt = &sh.cnt; fn.oflow = &sh.oflow; fn.pool = sh.pool;
                fn.sh64 = sh.sh64; fn.ired = sh.ired; fn.k = A.top_k;
                stream_row<E>(R, lrow, A.tma_l != 0, x0, x1, fn);
                uint64_t kth;
                const int keep = fn.finish(kth);
                const uint32_t bad = block_or(fn.bad, reinterpret_cast<uint32_t*>(sh.red));
                const int wr = keep < A.cap_p ? keep : A.cap_p;
                for (int i = threadIdx.x; i < wr; i += kThreads) __stcg(pk + i, sh.cand[i]);
                if (threadIdx.x == 0) {
                    uint32_t f = bad ? kPfBad : 0u;
                    if (sh.oflow || keep > A.cap_p) f |= kPfOverflow;
                    ph->flags = f;
                    ph->cnt = wr;
                    ph->kth = kth;
                    ph->vmax = keep ? ckey_val(sh.cand[0]) : -kInf;
                }
            } else {
                SumExpFn<E> fn;
                fn.c = A.c2;
                stream_row<E>(R, lrow, A.tma_l != 0, x0, x1, fn);
                // fold per-thread (m_t, s_t) into the slice max and sum
                const uint64_t mk = block_max_u64(static_cast<uint64_t>(fkey(fn.m)), reinterpret_cast<uint64_t*>(sh.red));
                const float ms = fkey_inv(static_cast<uint32_t>(mk));
                float sc = 0.f;
                if (fn.s > 0.f) sc = fn.s * ex2((fn.m - ms) * A.c2);
                const double tot = block_sum_d(static_cast<double>(sc), sh.red);
                const uint32_t bad = block_or(fn.bad, reinterpret_cast<uint32_t*>(sh.red));
                if (threadIdx.x == 0) {
                    ph->flags = bad ? kPfBad : 0u;
                    ph->cnt = 0;
                    ph->vmax = ms;
                    ph->sum = tot;
                }
            }
        } else if (kind == kResid) {
            const ReqState* rs = &A.W.req[b];
            ResidFn<E> fn;
            fn.m = static_cast<float>(__ldcg(&rs->m));
            fn.c = A.c2;
            fn.invZ = static_cast<float>(1.0 / __ldcg(&rs->Z));
            stream_row2<E>(R, chain_lrow<E>(A, b, row), chain_qrow(A, b, row),
                           (A.tma_l && A.tma_q), x0, x1, fn);
            const double rsum = block_sum_d(static_cast<double>(fn.r), sh.red);
            const double psum = block_sum_d(static_cast<double>(fn.pw), sh.red);
            if (threadIdx.x == 0) {
                ph->flags = 0;
                ph->sum = rsum;
                ph->sum2 = psum;
            }
        }
        if (arrive(A.W, b, A.S, &sh.last)) {
            const int st = initial ? 0 : __ldcg(&A.W.req[b].status);
            if (kind == kInvalid) {
                chain_finish(A, b, 0, -1, 16);
            } else if constexpr (kTopk) {
                combine_topk<E, kCap>(A, R, sh, b, row, kind, st);
            } else {
                combine_full<E, kCap>(A, sh, b, row, kind, st);
            }
            __syncthreads();
        }
    }
    if (R.err) atomicOr(&A.W.ctrl->error, kErrWait);
}

template <class E, bool kTopk>
static size_t chain_smem_bytes() {
    constexpr int kCap = kThreads * E::kVec + 512;
    return kStages * kChunkBytes + sizeof(ChainSmem<kCap>);
}

template <class E, bool kTopk>
static cudaError_t chain_launch(const ChainArgs& A, int grid, cudaStream_t st) {
    const size_t smem = chain_smem_bytes<E, kTopk>();
    cudaError_t e = cudaFuncSetAttribute(chain_kernel<E, kTopk>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    chain_kernel<E, kTopk><<<grid, kThreads, smem, st>>>(A);
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
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_kernel<F32, true>, kThreads, smem); }
        else { cudaFuncSetAttribute(chain_kernel<F32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
               cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_kernel<F32, false>, kThreads, smem); }
    } else {
        if (topk) { cudaFuncSetAttribute(chain_kernel<BF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_kernel<BF16, true>, kThreads, smem); }
        else { cudaFuncSetAttribute(chain_kernel<BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
               cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_kernel<BF16, false>, kThreads, smem); }
    }
    return n;
}

cudaError_t chain_run(const ChainArgs& A, int grid, cudaStream_t st) {
    const bool topk = A.top_k > 0 && A.top_k < A.V;
    if (A.ldt == 0) return topk ? chain_launch<F32, true>(A, grid, st) : chain_launch<F32, false>(A, grid, st);
    return topk ? chain_launch<BF16, true>(A, grid, st) : chain_launch<BF16, false>(A, grid, st);
}

}  // namespace spec
