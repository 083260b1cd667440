// spec_chain.cu -- batched chain speculative sampling on the cluster engine.
//
// [SD-survey] = "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
// (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash, DDTree and
// DSpark), chzhyang.github.io.  §1 "what speculative decoding guarantees":
// position i accepts its drafted token y_i with probability
// min(1, p_i(y_i)/q_i(y_i)); the first rejection commits a token drawn from
// the normalised residual [p_i - q_i]_+; if every draft passes, a bonus token
// is drawn from p_{K+1}; temperature and top-k truncation are part of p.
//
// Jobs of one request (every CTA of the cluster streams its vocabulary slice
// of the row unless a job names one target CTA):
//   TK row i      top-k rows: every slice's candidates for the row's top-k
//                 set (behind a certified or hinted value filter); the combine
//                 selects the set S, forms Z on it and takes the accept test;
//                 a rejection draws the correction from [p - q]_+ on S (q is
//                 gathered at S), a bonus row draws from p on S
//   SE row i      untruncated rows (or a top-k row whose threshold is known
//                 and whose tied set is too large to list): per slice the max
//                 and the sum of the weights; the combine takes the accept test
//   RESID row i   after an SE rejection: per slice the residual mass
//   RESCAN        one CTA draws inside its slice (the combine found the slice
//                 whose cumulative mass crosses the target)
//   RADIX round   an exact radix select of the k-th largest value (4 rounds),
//                 for top-k rows whose candidates overflowed (massive ties)
// Rows past the first rejection are never touched.
#include "spec_chain.cuh"
#include "spec_select.cuh"

namespace spec {

enum ChainKind : int { kTk = 0, kSe = 1, kResid = 2, kRescan = 3, kRadix = 4 };
// Job fields per kind:
//   row            the row (draft position; K or k_b is the bonus row)
//   aux            TK/SE/RADIX: 1 when the row is the bonus row
//   hint           TK: filter hint (value key, 0 = none); SE/RESID/RESCAN: mask
//                  value key (0 = none); RADIX: the prefix found so far
//   aux2           RADIX: round (low byte) and the rank still sought (>> 8);
//                  RESCAN: weight mode (0: p weights, 1: [p - q]_+)
//   f[0..3]        RESID: m, 1/Z; RESCAN: m, 1/Z, target t (float-float)

// Combiner scratch: the gathered candidate keys, then the top-k set sorted
// by token (ids and float-float weights).
constexpr int kCombKeys = 1024;
constexpr int kCombSet = 512;
constexpr int kRegKeys = 4;        // gathered keys a combiner lane holds in registers (128 per warp)

struct ChainSmem {
    TopkSmem tk;                      // consumers: slice candidates (top-k rows)
    alignas(16) uint64_t list[kCombKeys];   // combiner: gathered keys
    int stok[kCombSet];               // combiner: S by token
    float sval[kCombSet];             // combiner: S's logits by token
    float2 swt[kCombSet];             // combiner: weights by token
    int bins[256];                    // consumers: radix histogram
    float2 red2[kWarps];
    int ired[kWarps + 4];
    int hist[64];
    uint32_t scratch[kWarps + 2];
    uint64_t sh64[4];
    float wm[kWarps];
    float2 ws[kWarps];
    float2 ws2[kWarps];
    uint32_t wb[kWarps];
    uint32_t last_hint;               // combiner: filter hint from this CTA's latest top-k row
    float tau_prev;                   // combiner: the k-th value of that row
    int tau_ok;                       // tau_prev holds one
    int nsel;                         // consumers: keys a slice reports
};

__device__ __forceinline__ int chain_k(const ChainArgs& A, int b) {
    return A.k_per_req ? A.k_per_req[b] : A.K;
}
// the uniform that drives a row's draw: u[b, k_b] (chain), u[b, depth] (tree)
__device__ __forceinline__ int draw_uidx(const ChainArgs& A, const Job& j) {
    return A.tree ? j.depth : chain_k(A, j.b);
}
template <class E>
__device__ __forceinline__ const void* chain_lrow(const ChainArgs& A, int b, int i) {
    const long long r = A.k_per_req && A.l_row_off ? static_cast<long long>(A.l_row_off[b] + i) * A.l_rs
                                                   : static_cast<long long>(b) * A.l_bs + static_cast<long long>(i) * A.l_rs;
    return static_cast<const unsigned char*>(A.logits) + r * E::kBytes;
}
__device__ __forceinline__ const float* chain_qrow(const ChainArgs& A, int b, int i) {
    const long long r = A.k_per_req && A.q_row_off ? static_cast<long long>(A.q_row_off[b] + i) * A.q_rs
                                                   : static_cast<long long>(b) * A.q_bs + static_cast<long long>(i) * A.q_rs;
    return A.q + r;
}
__device__ __forceinline__ float chain_u(const ChainArgs& A, int b, int i) {
    return A.uniforms[static_cast<long long>(b) * ((A.tree ? A.L : A.K) + 1) + i];
}

// ---------------------------------------------------------------------------
// combiner-warp steps (all 32 lanes)
// ---------------------------------------------------------------------------
// Commit the request: accepted drafts, then `last` (correction/bonus, or -1),
// then -1 padding.
__device__ Job chain_finish(const ChainArgs& A, int b, int n, int last, int st) {
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
    return job_done();
}

// The stochastic tree walk's outputs: path_nodes[b][1..depth] and
// out_tokens[b][0..depth-1] were written on the way.
__device__ Job tree_done(const ChainArgs& A, int b, int depth, int last, int st) {
    const int W = A.L + 1;
    const int l = threadIdx.x & 31;
    int* pn = A.path_nodes + static_cast<long long>(b) * W;
    int* ot = A.out_tokens + static_cast<long long>(b) * W;
    for (int i = l; i < W; i += 32) {
        if (i > depth) { pn[i] = -1; ot[i] = -1; }
        if (i == depth) ot[i] = last;
    }
    if (l == 0) {
        pn[0] = 0;
        A.num_accepted[b] = depth;
        A.status[b] = st;
    }
    __syncwarp();
    return job_done();
}

// The request ends at the job's row with `last` committed (or -1).
__device__ __forceinline__ Job finish_at(const ChainArgs& A, const Job& j, int last, int st) {
    return A.tree ? tree_done(A, j.b, j.depth, last, st) : chain_finish(A, j.b, j.row, last, st);
}

__device__ __forceinline__ void chain_diag(const ChainArgs& A, int b, int i, float py, float qy, float Z, float R) {
    if (!A.diag || (threadIdx.x & 31) != 0) return;
    float* d = A.diag + (static_cast<long long>(b) * (A.K + 1) + i) * 4;
    d[0] = py; d[1] = qy; d[2] = Z; d[3] = R;
}
__device__ __forceinline__ void chain_diag_R(const ChainArgs& A, int b, int i, float R) {
    if (!A.diag || (threadIdx.x & 31) != 0) return;
    A.diag[(static_cast<long long>(b) * (A.K + 1) + i) * 4 + 3] = R;
}

// The job that reads row `row` of request b (a bonus row when row == k_b;
// in a tree walk every row is drawn from).
// `y`: the row's drafted token when the caller already loaded it
__device__ __forceinline__ Job row_job(const ChainArgs& A, int b, int row, int st, uint32_t hint, int depth = 0,
                                       int y = kYUnknown) {
    Job j = make_job(b, row, A.top_k > 0 ? kTk : kSe, st);
    j.aux = (A.tree || row >= chain_k(A, b)) ? 1 : 0;
    j.hint = A.top_k > 0 ? hint : 0u;
    j.depth = depth;
    j.y = y;
    return j;
}

// The drafted token of a draft row and its logit and q, loaded by the
// combiner warp with loads issued where they stand (the values are used only
// at the accept test, after the selection work).  `yn`: the next row's drafted
// token, issued now for the next job of this request.
// When the job does not carry y (a request's first row), y is loaded first
// and the dependent loads wait until ready() (nothing before the accept test
// waits on them).
// a chain job whose combine inputs the combiner loaded ahead (aux2; the
// values in f[0..3], pad[0] and y)
constexpr int kPrefetched = 0x7e1ec7;

template <class E>
struct DraftLoads {
    int y, yn;
    float ly, qy;
    bool pend;
    __device__ __forceinline__ void from_job(const Job& job) {
        y = job.y; yn = job.pad[0]; ly = job.f[2]; qy = job.f[3];
        pend = false;
    }
    __device__ __forceinline__ void load_lq(const ChainArgs& A, int b, int row) {
        ly = -kInf;
        qy = 0.f;
        if (y >= 0 && y < A.V) {
            const unsigned char* lr = static_cast<const unsigned char*>(chain_lrow<E>(A, b, row));
            if (E::kBytes == 4) ly = __uint_as_float(ldg_now_u32(lr + 4ll * y));
            else ly = __uint_as_float(ldg_now_u16(lr + 2ll * y) << 16);
            qy = __uint_as_float(ldg_now_u32(chain_qrow(A, b, row) + y));
        }
    }
    __device__ __forceinline__ void issue(const ChainArgs& A, const Job& job, int kb) {
        const int b = job.b, row = job.row;
        const int* dr = A.draft + static_cast<long long>(b) * A.K;
        yn = (row + 1 < kb) ? static_cast<int>(ldg_now_u32(dr + row + 1)) : kYUnknown;
        pend = job.y == kYUnknown;
        if (pend) {
            y = static_cast<int>(ldg_now_u32(dr + row));
        } else {
            y = job.y;
            load_lq(A, b, row);
        }
    }
    __device__ __forceinline__ void ready(const ChainArgs& A, const Job& job) {
        if (pend) load_lq(A, job.b, job.row);
    }
};

// A row's draw x is known: the chain commits it; the tree walk looks it up
// among the node's children and goes on there, or commits it as the bonus.
__device__ Job draw_done(const ChainArgs& A, const Job& j, int x, int st, uint32_t hint) {
    if (!A.tree) return chain_finish(A, j.b, j.row, x, st);
    const int child = x >= 0 ? find_child_w(A.t_token, A.t_parent, A.t_nn, A.N, j.b, j.row, x) : -1;
    if (child < 0 || j.depth >= A.L) return tree_done(A, j.b, j.depth, x, st);
    if ((threadIdx.x & 31) == 0) {
        const int W = A.L + 1;
        A.out_tokens[static_cast<long long>(j.b) * W + j.depth] = x;
        A.path_nodes[static_cast<long long>(j.b) * W + j.depth + 1] = child;
    }
    __syncwarp();
    return row_job(A, j.b, child, st, hint, j.depth + 1);
}

// Acceptance of drafted y: u < p(y)/q(y).  With weights scaled by the
// normaliser, p(y) = e_y / Z, the test is e_y > u q Z (float-float; no
// division on this path).
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
// m: `margin` of the gap below tau (rows of one target differ little in tau;
// a hint above the next row's tau costs a re-read of that row, one far below
// it extra candidates).
// The next call's first rows take a wider margin: 0.5 gave about 650
// candidates per slice (13 k) on N(0, 3^2) rows of 151936, each costing a
// slow row end; 0.25 ran faster both there and on rows whose scale varies.
#ifndef SPEC_PERSIST_MARGIN
#define SPEC_PERSIST_MARGIN 0.25f
#endif
// Within a call 0.16 of the gap: at 0.08 the next row's k-th value fell
// below the hint often enough that the second passes cost more than the
// extra candidates of a lower filter (dflash 172 -> 158 us, dspark 172 ->
// 162 us; 0.12, 0.2 and 0.3 measured in between).
#ifndef SPEC_HINT_MARGIN
#define SPEC_HINT_MARGIN 0.16f
#endif
__device__ __forceinline__ uint32_t hint_from(float tau, float m, float margin) {
    const float h = tau - margin * (m - tau);
    return (h == h && h > -kInf) ? fkey(h) : 0u;
}

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

// ---------------------------------------------------------------------------
// combine of a top-k row.  Every slice reports its keys at or above its own
// k-th value, sorted descending (composite keys: value, then lower id
// first).  S -- every element whose value reaches the row's k-th largest
// value tau -- is a union of prefixes of those lists, and tau is the value of
// the key whose merged rank is k - 1: each key's rank is the sum over the
// lists of the keys greater than it, by binary search.
// ---------------------------------------------------------------------------

// entries of the descending list lst[0..m) greater than x, for a warp's
// kRegKeys keys at once (s0: a power of two, at least m / 2)
__device__ __forceinline__ void count_gt4(const uint64_t* lst, int m, int s0, const uint64_t (&x)[kRegKeys],
                                          int (&pos)[kRegKeys]) {
#pragma unroll
    for (int j = 0; j < kRegKeys; ++j) pos[j] = 0;
    for (int s = s0; s > 0; s >>= 1) {
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j) {
            const int np = pos[j] + s;
            if (np <= m && lst[np - 1] > x[j]) pos[j] = np;
        }
    }
}
__device__ __forceinline__ const uint64_t* slice_keys(const unsigned char* parts, int pb, int r) {
    return reinterpret_cast<const uint64_t*>(part_at(parts, pb, r) + 1);
}
// the list holding flattened entry f (offsets `off` in lanes 0..C-1)
__device__ __forceinline__ int list_of(int off, int C, int f) {
    int r = 0;
    for (int q = 1; q < C; ++q) r += __shfl_sync(0xffffffffu, off, q) <= f ? 1 : 0;
    return r;
}

template <class E>
__device__ __noinline__ Job combine_topk(const ChainArgs& A, const Geo& G, const Job job, const unsigned char* parts,
                                         ChainSmem& sm) {
    if ((threadIdx.x & 31) == 0) SPEC_TRACE_EV(18, job.b, job.row, 0);
    SPEC_TRACE_T(tc0);
    const int l = threadIdx.x & 31;
    const int C = G.C, pb = G.part_bytes;
    const int b = job.b, row = job.row, k = A.top_k;
    const bool bonus = job.aux != 0;
    int st = job.st;
    // the request's global inputs this combine needs: loaded by the combiner
    // while the row streamed, else issued first so that their latency
    // overlaps the selection below
    float uk, ur;
    DraftLoads<E> dl;
    if (job.aux2 == kPrefetched) {
        uk = job.f[0];
        ur = job.f[1];
        dl.from_job(job);
    } else {
        uk = __uint_as_float(ldg_now_u32(&A.uniforms[static_cast<long long>(b) * ((A.tree ? A.L : A.K) + 1) +
                                                      draw_uidx(A, job)]));
        ur = bonus ? 0.f : __uint_as_float(ldg_now_u32(&A.uniforms[static_cast<long long>(b) *
                                                                    ((A.tree ? A.L : A.K) + 1) + row]));
        if (!bonus) dl.issue(A, job, chain_k(A, b));
    }
    SPEC_TRACE_T(tcu);
    SPEC_TRACE_T(tca);
    // the slices' headers (value filters: the low key halves are zero)
    const uint32_t hb = smem_u32(parts) + static_cast<uint32_t>(l * pb);
    uint32_t flags = 0, vkey = 0, thk = 0;
    int cnt = 0;
    if (l < C) {
        flags = lds_u32(hb + offsetof(PartHdr, flags));
        vkey = fkey(__uint_as_float(lds_u32(hb + offsetof(PartHdr, vmax))));
        thk = hkey(lds_u64(hb + offsetof(PartHdr, kth)));
        cnt = static_cast<int>(lds_u32(hb + offsetof(PartHdr, cnt)));
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    const float vmax = fkey_inv(__reduce_max_sync(0xffffffffu, vkey));
    const uint32_t th = __reduce_max_sync(0xffffffffu, thk);
    SPEC_TRACE_T(tcb);
    if ((flags & kPfBad) || !(vmax > -kInf)) return finish_at(A, job, -1, st | 1);
    if (flags & kPfOverflow) {
        // massive ties: the exact k-th value by radix select
        Job j = make_job(b, row, kRadix, st);
        j.aux = bonus ? 1 : 0;
        j.aux2 = (k << 8);
        j.depth = job.depth;
        return j;
    }
    // the prefix of each list at or above the largest slice filter holds
    // every member of S in that slice (two lists are merged whole: the split
    // search below needs no common cut)
    int mr = 0;
    if (C == 2) {
        mr = l < C ? cnt : 0;
    } else {
        // keys of list l at or above th: a power-of-two search over at most
        // 512 keys (every lane runs it; lanes >= C count none)
        const int cl = l < C ? cnt : 0;
        const uint32_t lr = smem_u32(parts) + static_cast<uint32_t>((l < C ? l : 0) * pb + sizeof(PartHdr));
#pragma unroll
        for (int s = 256; s > 0; s >>= 1) {
            const int np = mr + s;
            const uint32_t hv = hkey(lds_u64(lr + 8u * static_cast<uint32_t>(max(min(np, cl), 1) - 1)));
            mr = (np <= cl && hv >= th) ? np : mr;
        }
        if (cl >= 512 && mr == 511 && hkey(lds_u64(lr + 8u * 511u)) >= th) mr = 512;
    }
    int n, off;
    if (C == 2) {
        const int c0 = __shfl_sync(0xffffffffu, mr, 0), c1 = __shfl_sync(0xffffffffu, mr, 1);
        n = c0 + c1;
        off = l == 0 ? 0 : (l == 1 ? c0 : n);
    } else {
        off = warp_exscan_i(mr, n);
    }
    const uint32_t lt = (1u << l) - 1u;
    if (n < k) {
        // a hinted slice filter sat above the row's k-th value: stream the row
        // again without a hint (certified filters always leave k keys; without
        // a hint this is unreachable, and the radix path decides)
        if (job.hint != 0u) return row_job(A, b, row, st, 0u, job.depth);
        Job j = make_job(b, row, kRadix, st);
        j.aux = bonus ? 1 : 0;
        j.aux2 = (k << 8);
        j.depth = job.depth;
        return j;
    }
    if (n > kCombKeys) {
        Job j = make_job(b, row, kRadix, st);
        j.aux = bonus ? 1 : 0;
        j.aux2 = (k << 8);
        j.depth = job.depth;
        return j;
    }
    SPEC_TRACE_T(tc1);
    // the key of merged rank k - 1; then S (every key whose value reaches
    // it): its size, Z = sum of e_x = 2^((l_x - m) c) over it (float-float),
    // and its keys into the list (for a draw)
    const uint32_t mmax = warp_max_u32(static_cast<uint32_t>(mr));
    const int s0 = 1 << (31 - __clz(mmax));
    const uint32_t kbase = smem_u32(parts) + static_cast<uint32_t>(sizeof(PartHdr));   // + r * pb: slice r's keys
    const float m = vmax, c2 = A.c2;
    uint64_t tauc = 0;
    uint32_t tau_key;
    int keep = 0;
    dfloat zp = df_make(0.f);
    if (C == 2 && n <= 32 * kRegKeys) {
        // two lists: the k largest keys are A[0, i) and B[0, k - i) for the
        // one split i with A[i-1] > B[k-i] and B[k-i-1] > A[i] (where those
        // entries exist; keys are distinct).  Every candidate split is tested
        // at once, one per lane (adjacent entries: no bank conflicts), and
        // the k-th largest key is the smaller of the two prefixes' last.
        const int mA = __shfl_sync(0xffffffffu, mr, 0), mB = __shfl_sync(0xffffffffu, mr, 1);
        uint64_t key[kRegKeys];
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j) {
            const int f = min(l + 32 * j, n - 1);
            const uint32_t a = f < mA ? kbase + static_cast<uint32_t>(f * 8)
                                      : kbase + static_cast<uint32_t>(pb + (f - mA) * 8);
            const uint64_t v = lds_u64(a);
            key[j] = l + 32 * j < n ? v : 0ull;
        }
        const int lo = max(0, k - mB), hi = min(k, mA);
        const uint32_t la = kbase, lb = kbase + static_cast<uint32_t>(pb);
        tauc = 0ull;
        for (int i0 = lo; i0 <= hi; i0 += 32) {
            const int i = min(i0 + l, hi), j = k - i;
            const uint64_t a1 = lds_u64(la + 8u * static_cast<uint32_t>(max(i - 1, 0)));
            const uint64_t a0 = lds_u64(la + 8u * static_cast<uint32_t>(min(i, max(mA - 1, 0))));
            const uint64_t b1 = lds_u64(lb + 8u * static_cast<uint32_t>(max(j - 1, 0)));
            const uint64_t b0 = lds_u64(lb + 8u * static_cast<uint32_t>(min(j, max(mB - 1, 0))));
            const bool ok = i0 + l <= hi && (i == 0 || j == mB || a1 > b0) && (j == 0 || i == mA || b1 > a0);
            const uint64_t cand = i == 0 ? b1 : (j == 0 ? a1 : (a1 < b1 ? a1 : b1));
            const uint32_t who = __ballot_sync(0xffffffffu, ok);
            if (who) {
                const int src = __ffs(who) - 1;
                const uint32_t tlo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(cand), src);
                const uint32_t thi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(cand >> 32), src);
                tauc = (static_cast<uint64_t>(thi) << 32) | tlo;
                break;
            }
        }
        tau_key = hkey(tauc);
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j) {
            const bool p = l + 32 * j < n && hkey(key[j]) >= tau_key;
            if (p) zp = df_add(zp, ex2((ckey_val(key[j]) - m) * c2));
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            if (p) sm.list[keep + __popc(bal & lt)] = key[j];
            keep += __popc(bal);
        }
    } else if (C <= 4 && n <= 32 * kRegKeys) {
        // every search of every key at once: lists q >= C are empty (offset n)
        int o[4], mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            o[q] = __shfl_sync(0xffffffffu, off, q);
            mq[q] = __shfl_sync(0xffffffffu, mr, q);
        }
        // every load unconditional (indices clamped into a list that exists),
        // so that each step's sixteen loads issue back to back
        uint64_t key[kRegKeys];
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j) {
            const int f = min(l + 32 * j, n - 1);
            const int r = (f >= o[1] ? 1 : 0) + (f >= o[2] ? 1 : 0) + (f >= o[3] ? 1 : 0);
            const int base = r == 0 ? 0 : (r == 1 ? o[1] : (r == 2 ? o[2] : o[3]));
            const uint64_t v = lds_u64(kbase + static_cast<uint32_t>(r * pb + (f - base) * 8));
            key[j] = l + 32 * j < n ? v : 0ull;
        }
        int pos[4][kRegKeys];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < kRegKeys; ++j) pos[q][j] = 0;
        uint32_t lbase[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) lbase[q] = kbase + static_cast<uint32_t>((q < C ? q : 0) * pb);
        for (int s = s0; s > 0; s >>= 1) {
            uint64_t v[4][kRegKeys];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < kRegKeys; ++j) {
                    const int idx = max(min(pos[q][j] + s, mq[q]), 1) - 1;
                    v[q][j] = lds_u64(lbase[q] + static_cast<uint32_t>(idx * 8));
                }
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < kRegKeys; ++j) {
                    const int np = pos[q][j] + s;
                    pos[q][j] = (np <= mq[q] && v[q][j] > key[j]) ? np : pos[q][j];
                }
        }
        // the one key of rank k - 1: its lane and slot by ballots
        int jt = -1;
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j)
            if (l + 32 * j < n && pos[0][j] + pos[1][j] + pos[2][j] + pos[3][j] == k - 1) jt = j;
        const uint32_t who = __ballot_sync(0xffffffffu, jt >= 0);
        const int src = who ? __ffs(who) - 1 : 0;
        uint64_t mine = 0;
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j) mine = jt == j ? key[j] : mine;
        const uint32_t tlo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(mine), src);
        const uint32_t thi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(mine >> 32), src);
        tauc = (static_cast<uint64_t>(thi) << 32) | tlo;
        tau_key = hkey(tauc);
#pragma unroll
        for (int j = 0; j < kRegKeys; ++j) {
            const bool p = l + 32 * j < n && hkey(key[j]) >= tau_key;
            if (p) zp = df_add(zp, ex2((ckey_val(key[j]) - m) * c2));
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            if (p) sm.list[keep + __popc(bal & lt)] = key[j];
            keep += __popc(bal);
        }
    } else {
        for (int f0 = 0; f0 < n; f0 += 32 * kRegKeys) {
            uint64_t key[kRegKeys];
            int rank[kRegKeys], pos[kRegKeys];
#pragma unroll
            for (int j = 0; j < kRegKeys; ++j) {
                const int f = f0 + l + 32 * j;
                const int r = list_of(off, C, f);
                const int base = __shfl_sync(0xffffffffu, off, r);
                key[j] = f < n ? lds_u64(kbase + static_cast<uint32_t>(r * pb + (f - base) * 8)) : 0ull;
                rank[j] = 0;
            }
            for (int q = 0; q < C; ++q) {
                const int mqq = __shfl_sync(0xffffffffu, mr, q);
                count_gt4(slice_keys(parts, pb, q), mqq, s0, key, pos);
#pragma unroll
                for (int j = 0; j < kRegKeys; ++j) rank[j] += pos[j];
            }
#pragma unroll
            for (int j = 0; j < kRegKeys; ++j)
                if (f0 + l + 32 * j < n && rank[j] == k - 1) tauc = key[j];
        }
        tauc = warp_max_u64(tauc);
        tau_key = hkey(tauc);
        for (int f0 = 0; f0 < n; f0 += 32) {
            const int f = f0 + l;
            const int r = list_of(off, C, f);
            const int base = __shfl_sync(0xffffffffu, off, r);
            const uint64_t key = f < n ? lds_u64(kbase + static_cast<uint32_t>(r * pb + (f - base) * 8)) : 0ull;
            const bool p = f < n && hkey(key) >= tau_key;
            if (p) zp = df_add(zp, ex2((ckey_val(key) - m) * c2));
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            if (p) sm.list[keep + __popc(bal & lt)] = key;
            keep += __popc(bal);
        }
    }
    const float tau = fkey_inv(tau_key);
    const dfloat Z = warp_sum_df(zp);
    __syncwarp();
    SPEC_TRACE_T(tc2);
    if (keep > kCombSet) {
        // a large tied set: the masked full-row passes, with the threshold known
        Job j = make_job(b, row, kSe, st);
        j.aux = bonus ? 1 : 0;
        j.hint = tau_key;
        j.depth = job.depth;
        return j;
    }
    // the next rows' filter hint (and, persisted, the next call's) -- only
    // while the rows keep their k-th value: this row's hint (if it had one)
    // sat less than the row's max-to-tau gap below tau, else tau moved less
    // than half that gap from the previous row this combiner saw.  Rows whose
    // scale or offset moves from row to row get no hint (their slices start
    // from a certified bound instead), so a stale hint costs no second pass.
    const float gap = m - tau;
    const bool steady = job.hint != 0u ? key_to_thr(job.hint) >= tau - gap
                                       : (sm.tau_ok && fabsf(tau - sm.tau_prev) <= 0.5f * gap);
    const uint32_t hint = steady ? hint_from(tau, m, SPEC_HINT_MARGIN) : 0u;
    if (l == 0) {
        sm.last_hint = hint;
        sm.tau_prev = tau;
        sm.tau_ok = tau == tau && tau > -kInf && m < kInf;
        // for the next call's first rows, with a wider margin (another call's
        // rows may sit lower); one 16-byte store
        const uint32_t hw = steady ? hint_from(tau, m, SPEC_PERSIST_MARGIN) : 0u;
        __stcg(reinterpret_cast<uint4*>(A.E.W.ctrl->persist),
               make_uint4(kPersistTag, hw, static_cast<uint32_t>(A.V), static_cast<uint32_t>(A.top_k)));
    }
    auto prob = [&](float e) { return static_cast<float>(static_cast<double>(e) / df_to_d(Z)); };   // diagnostics
    float ey = 0.f, qy = 0.f;
    if (!bonus) {
        dl.ready(A, job);
        const int y = dl.y;
        const float ly = dl.ly;
        qy = dl.qy;
        ey = (y >= 0 && y < A.V && fkey(ly) >= tau_key) ? ex2((ly - m) * c2) : 0.f;
        const bool acc = chain_accept_z(A, y, ey, qy, Z, ur, st);
#ifdef SPEC_TRACE
        SPEC_TRACE_T(tc3);
        if (l == 0) {
            SPEC_TRACE_EV(11, n, keep, static_cast<int>(tc1 - tc0));
            SPEC_TRACE_EV(12, static_cast<int>(tc2 - tc1), static_cast<int>(tc3 - tc2), 0);
            SPEC_TRACE_EV(22, static_cast<int>(tca - tc0), static_cast<int>(tcb - tc0), static_cast<int>(tc1 - tc0));
            SPEC_TRACE_EV(23, static_cast<int>(tcu - tc0), 0, 0);
        }
#endif
        if (acc) {
            if (A.diag) chain_diag(A, b, row, prob(ey), qy, Z.hi, 0.f);
            if (l == 0) SPEC_TRACE_EV(19, b, row, 0);
            return row_job(A, b, row + 1, st, hint, 0, dl.yn);
        }
    }
    // a draw on S (the residual at a rejection, p at the bonus row): S sorted
    // by token id (ids in S are distinct), each member's rank the number of
    // smaller ids, counted over shuffles (or shared memory beyond 64)
    if (keep <= 64) {
        const uint64_t k0 = l < keep ? sm.list[l] : 0ull, k1 = l + 32 < keep ? sm.list[l + 32] : 0ull;
        const int t0 = l < keep ? ckey_idx(k0) : 0x7fffffff;
        const int t1 = l + 32 < keep ? ckey_idx(k1) : 0x7fffffff;
        int r0 = 0, r1 = 0;
#pragma unroll 8
        for (int o = 0; o < 32; ++o) {
            const int a = __shfl_sync(0xffffffffu, t0, o), c = __shfl_sync(0xffffffffu, t1, o);
            r0 += (a < t0) + (c < t0);
            r1 += (a < t1) + (c < t1);
        }
        __syncwarp();
        if (l < keep) { sm.stok[r0] = t0; sm.sval[r0] = ckey_val(k0); }
        if (l + 32 < keep) { sm.stok[r1] = t1; sm.sval[r1] = ckey_val(k1); }
    } else {
        for (int i = l; i < keep; i += 32) {
            const uint64_t key = sm.list[i];
            const int x = ckey_idx(key);
            int r = 0;
            for (int t = 0; t < keep; ++t) r += ckey_idx(sm.list[t]) < x;
            sm.stok[r] = x;
            sm.sval[r] = ckey_val(key);
        }
    }
    __syncwarp();
    if (!bonus) {
        // residual [p - q]_+ lives on S (p = 0 outside it)
        const float* qrow = chain_qrow(A, b, row);
        dfloat rp = df_make(0.f);
        for (int i = l; i < keep; i += 32) {
            const float qx = __ldcg(qrow + sm.stok[i]);
            const float e = ex2((sm.sval[i] - m) * c2);
            const dfloat d = df_add(df_make(e), df_neg(df_mul(qx, Z)));
            const dfloat w = d.hi > 0.f ? d : df_make(0.f);
            sm.swt[i] = make_float2(w.hi, w.lo);
            rp = df_add(rp, w);
        }
        dfloat R = warp_sum_df(rp);
        __syncwarp();
        if (!(R.hi > 0.f)) {
            st |= 4;
            for (int i = l; i < keep; i += 32) sm.swt[i] = make_float2(ex2((sm.sval[i] - m) * c2), 0.f);
            __syncwarp();
            R = Z;
        }
        const int x = warp_icdf_pairs(sm.stok, sm.swt, keep, df_mul(uk, R));
        chain_diag(A, b, row, prob(ey), qy, Z.hi, (st & 4) ? 0.f : static_cast<float>(df_to_d(R) / df_to_d(Z)));
        return chain_finish(A, b, row, x, st);
    }
    // bonus row: draw from p on S
    for (int i = l; i < keep; i += 32) sm.swt[i] = make_float2(ex2((sm.sval[i] - m) * c2), 0.f);
    __syncwarp();
    const int x = warp_icdf_pairs(sm.stok, sm.swt, keep, df_mul(uk, Z));
    float px = 0.f;
    for (int i = l; i < keep; i += 32)
        if (sm.stok[i] == x) px = prob(sm.swt[i].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) px = fmaxf(px, __shfl_xor_sync(0xffffffffu, px, o));
    if (!A.tree) chain_diag(A, b, row, px, 0.f, Z.hi, 0.f);
    return draw_done(A, job, x, st, hint);
}

// ---------------------------------------------------------------------------
// combine of a sum-exp row (untruncated, or masked at a known threshold)
// ---------------------------------------------------------------------------
template <class E>
__device__ __noinline__ Job combine_se(const ChainArgs& A, const Geo& G, const Job job, const unsigned char* parts,
                                       ChainSmem& sm) {
    const int l = threadIdx.x & 31;
    const int C = G.C, pb = G.part_bytes;
    const int b = job.b, row = job.row;
    const bool bonus = job.aux != 0;
    const uint32_t mask = job.hint;
    int st = job.st;
    const float c2 = A.c2;
    const bool pre = job.aux2 == kPrefetched;
    DraftLoads<E> dl;
    if (pre) dl.from_job(job);
    else if (!bonus) dl.issue(A, job, chain_k(A, b));
    uint32_t flags = 0;
    float vm = -kInf;
    dfloat sv = df_make(0.f);
    if (l < C) {
        const PartHdr* h = part_at(parts, pb, l);
        flags = h->flags; vm = h->vmax; sv = df_of(h->sum);
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    float m = vm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((flags & kPfBad) || !(m > -kInf)) return finish_at(A, job, -1, st | 1);
    dfloat zv = df_make(0.f);
    if (l < C && sv.hi > 0.f) zv = df_mul(ex2((vm - m) * c2), sv);
    const dfloat Z = warp_sum_df(zv);
    const float uk = pre ? job.f[0] : chain_u(A, b, draw_uidx(A, job));
    if (!bonus) {
        dl.ready(A, job);
        const int y = dl.y;
        const float ly = dl.ly, qy = dl.qy;
        const float ey = (y >= 0 && y < A.V && fkey(ly) >= mask) ? ex2((ly - m) * c2) : 0.f;
        const bool acc = chain_accept_z(A, y, ey, qy, Z, pre ? job.f[1] : chain_u(A, b, row), st);
        chain_diag(A, b, row, static_cast<float>(static_cast<double>(ey) / df_to_d(Z)), qy, Z.hi, 0.f);
        if (acc) return row_job(A, b, row + 1, st, sm.last_hint, 0, dl.yn);
        // the residual pass: every slice's [p - q]_+ mass with this row's m and Z
        Job j = make_job(b, row, kResid, st);
        j.hint = mask;
        j.f[0] = m;
        j.f[1] = __frcp_rn(Z.hi);
        return j;
    }
    // bonus: the slice where the cumulative p mass crosses u Z, then a rescan there
    const dfloat t = df_mul(uk, Z);
    dfloat before;
    const int s = find_slice_w(C, zv, t, before);
    const dfloat tr = df_add(t, df_neg(before));
    Job j = make_job(b, row, kRescan, st);
    j.target = s;
    j.hint = mask;
    j.aux = 1;                       // bonus row
    j.aux2 = 0;                      // p weights
    j.f[0] = m; j.f[1] = 0.f; j.f[2] = tr.hi; j.f[3] = tr.lo;
    j.depth = job.depth;
    if (!A.tree) chain_diag(A, b, row, 0.f, 0.f, Z.hi, 0.f);
    return j;
}

__device__ __noinline__ Job combine_resid(const ChainArgs& A, const Geo& G, const Job job, const unsigned char* parts) {
    const int l = threadIdx.x & 31;
    const int C = G.C, pb = G.part_bytes;
    const int b = job.b, row = job.row;
    int st = job.st;
    const int kb = chain_k(A, b);
    dfloat rv = df_make(0.f), pv = df_make(0.f);
    if (l < C) {
        const PartHdr* h = part_at(parts, pb, l);
        rv = df_of(h->sum);
        pv = df_of(h->sum2);
    }
    const dfloat R = warp_sum_df(rv), Pm = warp_sum_df(pv);
    const float uk = chain_u(A, b, kb);
    dfloat t, before;
    int s, wmode;
    if (R.hi > 0.f) {
        t = df_mul(uk, R);
        s = find_slice_w(C, rv, t, before);
        wmode = 1;
    } else {
        st |= 4;
        t = df_mul(uk, Pm);
        s = find_slice_w(C, pv, t, before);
        wmode = 0;
    }
    chain_diag_R(A, b, row, (st & 4) ? 0.f : static_cast<float>(df_to_d(R)));
    const dfloat tr = df_add(t, df_neg(before));
    Job j = make_job(b, row, kRescan, st);
    j.target = s;
    j.hint = job.hint;
    j.aux = 0;
    j.aux2 = wmode;
    j.f[0] = job.f[0]; j.f[1] = job.f[1]; j.f[2] = tr.hi; j.f[3] = tr.lo;
    return j;
}

template <class E>
__device__ __noinline__ Job combine_rescan(const ChainArgs& A, const Job job, const unsigned char* parts, int pb,
                                           uint32_t hint) {
    const PartHdr* h = part_at(parts, pb, job.target);
    const int x = h->tok;
    const int b = job.b, row = job.row;
    if (job.aux != 0) {
        if (A.diag && !A.tree && (threadIdx.x & 31) == 0 && x >= 0 && x < A.V) {
        // bonus row: p(x) = e_x / Z, with Z as the SE combine recorded it
            float* d = A.diag + (static_cast<long long>(b) * (A.K + 1) + row) * 4;
            const float e = ex2((E::load(chain_lrow<E>(A, b, row), x) - job.f[0]) * A.c2);
            d[0] = static_cast<float>(static_cast<double>(e) / static_cast<double>(d[2]));
        }
        __syncwarp();
        return draw_done(A, job, x, job.st, hint);
    }
    return chain_finish(A, b, row, x, job.st);
}

__device__ __noinline__ Job combine_radix(const ChainArgs& A, const Geo& G, const Job job, const unsigned char* parts) {
    const int l = threadIdx.x & 31;
    const int C = G.C, pb = G.part_bytes;
    const int round = job.aux2 & 0xff;
    int want = job.aux2 >> 8;                 // rank sought among keys with this prefix
    uint32_t flags = 0;
    if (l < C) flags = part_at(parts, pb, l)->flags;
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (flags & kPfBad) return finish_at(A, job, -1, job.st | 1);
    // bins summed over the slices; lane l holds digits 8l .. 8l+7
    int cnt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int c = 0;
        for (int r = 0; r < C; ++r) c += reinterpret_cast<const int*>(part_at(parts, pb, r) + 1)[8 * l + j];
        cnt[j] = c;
    }
    // digits from the top: the one where the running count reaches `want`
    int lane_tot = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) lane_tot += cnt[j];
    int above = 0;   // keys in higher lanes (larger digits)
    {
        int suf = lane_tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_down_sync(0xffffffffu, suf, o);
            if (l + o < 32) suf += t;
        }
        above = suf - lane_tot;
    }
    int digit = -1, rem = 0;
    {
        int run = above;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
            if (digit < 0 && run + cnt[j] >= want) { digit = 8 * l + j; rem = want - run; }
            run += cnt[j];
        }
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, digit >= 0);
    const int src = bal ? 31 - __clz(bal) : 0;   // the highest lane that reached it holds the digit
    digit = __shfl_sync(0xffffffffu, digit, src);
    rem = __shfl_sync(0xffffffffu, rem, src);
    if (digit < 0) { digit = 0; rem = 1; }        // unreachable: fewer than k keys in the row
    const uint32_t prefix = (job.hint << 8) | static_cast<uint32_t>(digit);
    if (round < 3) {
        Job j = make_job(job.b, job.row, kRadix, job.st);
        j.aux = job.aux;
        j.hint = prefix;
        j.aux2 = (rem << 8) | (round + 1);
        j.depth = job.depth;
        return j;
    }
    // the exact threshold: the masked sum-exp passes take it from here
    Job j = make_job(job.b, job.row, kSe, job.st);
    j.aux = job.aux;
    j.hint = prefix;
    j.depth = job.depth;
    return j;
}

// A slice's report of a top-k row (all consumers): the keys src[0..n) at or
// above the slice filter F, sorted descending into dst by rank (the number of
// greater keys; keys are distinct), then cut after the last key whose value
// reaches the slice's k-th largest value -- no element below that value can
// be among the row's top k.  F is raised to that value.  Returns the count.
static_assert(TopkSmem::kSlots * kThreads >= 512, "the slots hold a slice's reported keys");
__device__ int slice_sort_trim(const uint64_t* src, int n, uint64_t& F, int k, uint64_t* dst, int* nsel) {
    if (threadIdx.x == 0) *nsel = 0;
    csync();   // src complete, the count zeroed
    int mine = 0;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint64_t x = src[i];
        if (x < F) continue;
        int r = 0;
#pragma unroll 8
        for (int j = 0; j < n; ++j) r += src[j] > x ? 1 : 0;   // greater keys reach F as well
        dst[r] = x;
        ++mine;
    }
    if (mine) atomicAdd(nsel, mine);
    csync();
    const int nf = *nsel;
    if (nf < k) return nf;   // a hint above the slice's k-th value: every key counts
    const uint32_t vk = hkey(dst[k - 1]);
    int lo = k, hi = nf;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (hkey(dst[mid]) >= vk) lo = mid + 1; else hi = mid;
    }
    const uint64_t fk = static_cast<uint64_t>(vk) << 32;
    if (fk > F) F = fk;
    return lo;
}

// The inverse CDF of a draw inside this CTA's slice (a RESCAN job; all
// consumers): the smallest x with C(x) > t, C the inclusive prefix of the
// weights in ascending x (residual [e / Z - q]_+ when aux2 == 1, else e), in
// float-float; if rounding leaves no crossing, the last x with a positive
// weight (or the slice start).  The slice streams through the ring like any
// row; each chunk is scanned in shared memory with every thread on a run of
// consecutive elements: the run's sum, a block exclusive scan, and the one
// thread whose run crosses t walks it again.  Chunks after the crossing are
// released unread.  Returns kIcdfDead when a chunk wait gave up.
constexpr int kIcdfDead = -0x7ffffff0;
template <class E>
__device__ int consume_icdf(const ChainArgs& A, const Pipe& P, uint32_t& seq, const StreamPlan& p, bool tma, int x0,
                            const Job& j, ChainSmem& sm) {
    const float m = j.f[0], c2 = A.c2, invZ = j.f[1];
    const float thr = j.hint ? key_to_thr(j.hint) : -kInf;
    const dfloat t{j.f[2], j.f[3]};
    const bool resid = j.aux2 == 1;
    bool dead = false;
    int found = 0x7fffffff, last_pos = -1;
    dfloat base = df_make(0.f);
    for (int c = 0; c < p.nch; ++c, ++seq) {
        const bool have = take_chunk(P, seq, tma, dead, p, c);
        // CTA-uniform (the barriers below): a warp whose wait gave up
        // contributes nothing
        if (found == 0x7fffffff) {
            const unsigned char* sm_l = P.slot(P.stage(seq));
            const float* sm_q = reinterpret_cast<const float*>(sm_l + p.ce * E::kBytes);
            const int ne = min(p.ce, p.n - c * p.ce);
            // bytes past the 16-byte-multiple prefix were not copied by TMA
            const int l_in = tma ? ((ne * E::kBytes) & ~15) / E::kBytes : ne;
            const int q_in = tma ? ((ne * 4) & ~15) / 4 : ne;
            const float* gq = resid ? reinterpret_cast<const float*>(p.src1) + static_cast<long long>(c) * p.ce : nullptr;
            auto weight = [&](int i) -> float {
                const float lv = i < l_in ? E::load(sm_l, i) : E::load(p.src0, static_cast<long long>(c) * p.ce + i);
                const float e = lv >= thr ? ex2((lv - m) * c2) : 0.f;
                if (!resid) return e;
                const float qv = i < q_in ? sm_q[i] : gq[i];
                const float d = e * invZ - qv;
                return d > 0.f ? d : 0.f;
            };
            const int per = (ne + kThreads - 1) / kThreads;
            const int i0 = threadIdx.x * per, i1 = have ? min(ne, i0 + per) : i0;
            dfloat loc = df_make(0.f);
            int lp = -1;
            for (int i = i0; i < i1; ++i) {
                const float w = weight(i);
                loc = df_add(loc, w);
                if (w > 0.f) lp = i;
            }
            dfloat tot;
            const dfloat c0 = df_add(base, block_exscan_df(loc, sm.red2, tot));
            int mine = 0x7fffffff;
            if (loc.hi > 0.f && df_gt(df_add(c0, loc), t)) {
                dfloat cc = c0;
                for (int i = i0; i < i1; ++i) {
                    const float w = weight(i);
                    cc = df_add(cc, w);
                    if (w > 0.f && df_gt(cc, t)) { mine = i; break; }
                }
            }
            if (threadIdx.x == 0) { sm.ired[0] = 0x7fffffff; sm.ired[1] = -1; }
            csync();
            if (mine != 0x7fffffff) atomicMin(&sm.ired[0], mine);
            if (lp >= 0) atomicMax(&sm.ired[1], lp);
            csync();
            const int cx0 = x0 + c * p.ce;
            if (sm.ired[0] != 0x7fffffff) found = cx0 + sm.ired[0];
            if (sm.ired[1] >= 0) last_pos = cx0 + sm.ired[1];
            base = df_add(base, tot);
            csync();   // ired is read before the next chunk resets it
        }
        release_chunk(P, seq, tma, dead);
    }
    if (csync_or(dead)) return kIcdfDead;
    return found != 0x7fffffff ? found : (last_pos >= 0 ? last_pos : x0);
}

// ---------------------------------------------------------------------------
// the op
// ---------------------------------------------------------------------------
template <class E, bool kTopk>
struct ChainOp {
    using Args = ChainArgs;
    using Smem = ChainSmem;

    __device__ static int batch(const Args& A) { return A.B; }
    __device__ static bool tma(const Args& A) { return A.tma_l && (kTopk || A.K == 0 || A.tma_q); }
    // A chain row's combine inputs, loaded by the combiner while the row
    // streams (right after the job was posted): the row's uniforms, its
    // drafted token and the next row's, the token's logit and q.  They go to
    // the combiner's own copy of the job (the posted copies are not touched),
    // so the combine starts without a global load.
    __device__ static void prefetch(const Args& A, const Geo&, Job& j, Smem&) {
        if (A.tree || j.b < 0 || (j.kind != kTk && j.kind != kSe)) return;
        if ((threadIdx.x & 31) == 0) {
            const int b = j.b, row = j.row;
            const int kb = chain_k(A, b);
            const long long ub = static_cast<long long>(b) * (A.K + 1);
            const bool bonus = j.aux != 0;
            const float uk = A.uniforms[ub + kb];
            const float ur = bonus ? 0.f : A.uniforms[ub + row];
            int y = kYUnknown, yn = kYUnknown;
            float ly = -kInf, qy = 0.f;
            if (!bonus) {
                const int* dr = A.draft + static_cast<long long>(b) * A.K;
                yn = row + 1 < kb ? dr[row + 1] : kYUnknown;
                y = j.y != kYUnknown ? j.y : dr[row];
                if (y >= 0 && y < A.V) {
                    ly = E::load(chain_lrow<E>(A, b, row), y);
                    qy = chain_qrow(A, b, row)[y];
                }
            }
            j.f[0] = uk; j.f[1] = ur; j.f[2] = ly; j.f[3] = qy;
            j.pad[0] = yn;
            j.y = y;
            j.aux2 = kPrefetched;
        }
        __syncwarp();
    }
    __device__ static void init_smem(const Args& A, const Geo&, Smem& sm) {
        if (threadIdx.x == 0) {
            topk_smem_init(sm.tk);
            // the previous call's hint on this workspace, for the same
            // vocabulary and top-k: the first rows' filter until a row of
            // this call gives a better one
            uint32_t h = 0;
            if (kTopk) {
                const uint4 ps = __ldcg(reinterpret_cast<const uint4*>(A.E.W.ctrl->persist));
                if (ps.x == kPersistTag && ps.z == static_cast<uint32_t>(A.V) &&
                    ps.w == static_cast<uint32_t>(A.top_k))
                    h = ps.y;
            }
            sm.last_hint = h;
            sm.tau_prev = 0.f;
            sm.tau_ok = 0;
        }
    }
    __device__ static Job first(const Args& A, const Geo&, int b, Smem& sm) {
        const int kb = A.tree ? 0 : chain_k(A, b);
        if (kb < 0 || kb > A.K) return chain_finish(A, b, 0, -1, 16);
        return row_job(A, b, 0, 0, sm.last_hint);
    }
    __device__ static StreamPlan plan(const Args& A, const Geo& G, const Job& j) {
        const int x0 = slice_x0(G, G.rank), x1 = slice_x1(G, G.rank, A.V);
        switch (j.kind) {
            case kTk: case kSe: case kRadix:
                return plan_single(chain_lrow<E>(A, j.b, j.row), E::kBytes, x0, x1, G.chunk);
            case kResid:
                return plan_dual(chain_lrow<E>(A, j.b, j.row), E::kBytes, chain_qrow(A, j.b, j.row), x0, x1, G.chunk);
            case kRescan:
                // the target CTA streams its slice (logits, and q for residual weights)
                return j.aux2 == 1 ? plan_dual(chain_lrow<E>(A, j.b, j.row), E::kBytes, chain_qrow(A, j.b, j.row), x0,
                                               x1, G.chunk)
                                   : plan_single(chain_lrow<E>(A, j.b, j.row), E::kBytes, x0, x1, G.chunk);
            default:
                return plan_none();
        }
    }

    // consumers: this CTA's slice of the job -> the partial in `out`
    __device__ static int consume(const Args& A, const Geo& G, const Pipe& P, uint32_t& seq, bool tma, const Job& j,
                                  Smem& sm, unsigned char* out) {
        PartHdr* ph = reinterpret_cast<PartHdr*>(out);
        uint64_t* pk = reinterpret_cast<uint64_t*>(ph + 1);
        const int x0 = slice_x0(G, G.rank);
        const StreamPlan plan = ChainOp::plan(A, G, j);
        if (threadIdx.x == 0) {
            ph->flags = 0; ph->cnt = 0; ph->tok = -1; ph->kth = 0; ph->vmax = -kInf; ph->hasy = 0;
            ph->sum = make_float2(0.f, 0.f); ph->sum2 = make_float2(0.f, 0.f); ph->ly = -kInf; ph->qy = 0.f;
        }
        int nkeys = 0;
        if (j.kind == kTk || j.kind == kSe) {
            // (the drafted token's logit and q are the combiner's own loads)
            if (kTopk && j.kind == kTk) {
                TopkHistFn<E, true> fn;
                fn.init(&sm.tk, A.top_k, j.hint, seq + 1u);   // every consumer holds the same seq
                if (!consume_row<E>(P, seq, plan, tma, x0, fn)) return -1;
                SPEC_TRACE_T(tp0);
                fn.publish();
                csync();
                int tot;
                uint64_t F;
                uint32_t fl;
                float vm;
                fn.summary(tot, F, fl, vm);
                SPEC_TRACE_T(tp1);
                const uint32_t bad = (fl >> 1) & 1u;
                uint32_t oflow = fl & 1u;
                int n = tot;
                const uint64_t* src = nullptr;
                if (!bad && !oflow && tot <= A.cap_p) {
                    // every warp's keys at its offset, into the (flushed) slots
                    uint64_t* tmp = &sm.tk.slot[0][0];
                    fn.write_keys(tmp);
                    src = tmp;
                } else if (!bad && !oflow) {
                    // too many: the certified bound over every candidate, repeated
                    // until it stops rising (then it is the exact k-th value)
                    uint32_t o2, b2;
                    float vm2;
                    n = fn.finish(F, o2, b2, vm2);
                    uint64_t* list = sm.tk.cand;
                    for (int it = 0; it < 8 && n > A.cap_p; ++it) {
                        bool cert;
                        const uint32_t F2 = hist_bound_list(list, n, A.top_k, hkey(F), sm.hist, sm.scratch, cert);
                        if (!(cert && F2 > hkey(F))) break;
                        n = compact_list(list, n, F2, sm.ired);
                        F = static_cast<uint64_t>(F2) << 32;
                    }
                    if (n > A.cap_p) oflow = 1;   // ties at the k-th value: the combine takes the radix path
                    else src = list;
                }
                SPEC_TRACE_T(tp2);
                if (oflow || bad) n = 0;
                else n = slice_sort_trim(src, n, F, A.top_k, pk, &sm.nsel);
                nkeys = n;
                if (threadIdx.x == 0) {
                    ph->flags = (bad ? kPfBad : 0u) | (oflow ? kPfOverflow : 0u) | (j.hint ? kPfHinted : 0u);
                    ph->cnt = n;
                    ph->kth = F;
                    ph->vmax = vm;
                    SPEC_TRACE_EV(27, static_cast<int>(tp1 - tp0), static_cast<int>(tp2 - tp1),
                                  static_cast<int>(clock64() - tp2));
                    SPEC_TRACE_EV(28, tot, n, static_cast<int>(j.hint));
                }
            } else {
                // sum-exp (masked at the job's threshold when it carries one)
                const uint32_t mask = j.hint;
                auto run = [&](auto& fn) -> bool {
                    fn.c = A.c2;
                    if (!consume_row<E>(P, seq, plan, tma, x0, fn)) return false;
                    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
                    float wm = fn.m;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
                    const float sc = (fn.s > 0.f) ? fn.s * ex2((fn.m - wm) * A.c2) : 0.f;
                    const dfloat wsd = warp_sum_df(df_make(sc));
                    float wv = fn.vmx;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) wv = max_nan(wv, __shfl_xor_sync(0xffffffffu, wv, o));
                    const uint32_t wb = __reduce_or_sync(0xffffffffu, fn.bad_flag());
                    if (lane == 0) { sm.wm[w] = wm; sm.ws[w] = make_float2(wsd.hi, wsd.lo); sm.wb[w] = wb; sm.ws2[w].x = wv; }
                    csync();
                    if (threadIdx.x == 0) {
                        float ms = -kInf, vx = -kInf;
                        uint32_t bad = 0;
                        for (int q = 0; q < kWarps; ++q) { ms = fmaxf(ms, sm.wm[q]); bad |= sm.wb[q]; vx = max_nan(vx, sm.ws2[q].x); }
                        dfloat tot = df_make(0.f);
                        for (int q = 0; q < kWarps; ++q)
                            if (sm.ws[q].x > 0.f) tot = df_add(tot, df_mul(ex2((sm.wm[q] - ms) * A.c2), df_of(sm.ws[q])));
                        ph->flags = bad ? kPfBad : 0u;
                        ph->vmax = bad ? vx : ms;
                        ph->sum = make_float2(tot.hi, tot.lo);
                        }
                    return true;
                };
                bool ok;
                if (mask == 0u) {
                    SumExpFn<E, false> fn;
                    ok = run(fn);
                } else {
                    SumExpFn<E, true> fn;
                    fn.thr = key_to_thr(mask);
                    ok = run(fn);
                }
                if (!ok) return -1;
            }
        } else if (j.kind == kResid) {
            ResidFn<E> fn;
            fn.m = j.f[0];
            fn.c = A.c2;
            fn.invZ = j.f[1];
            fn.thr = j.hint ? key_to_thr(j.hint) : -kInf;
            if (!consume_row2<E>(P, seq, plan, tma, x0, fn)) return -1;
            const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
            const dfloat wr = warp_sum_df(df_make(fn.r));
            const dfloat wp = warp_sum_df(df_make(fn.pw));
            if (lane == 0) { sm.ws[w] = make_float2(wr.hi, wr.lo); sm.ws2[w] = make_float2(wp.hi, wp.lo); }
            csync();
            if (threadIdx.x == 0) {
                dfloat rsum = df_make(0.f), psum = df_make(0.f);
                for (int q = 0; q < kWarps; ++q) { rsum = df_add(rsum, df_of(sm.ws[q])); psum = df_add(psum, df_of(sm.ws2[q])); }
                ph->sum = make_float2(rsum.hi, rsum.lo);
                ph->sum2 = make_float2(psum.hi, psum.lo);
            }
        } else if (j.kind == kRescan) {
            // the inverse CDF inside this slice, streamed through the ring
            const int x = consume_icdf<E>(A, P, seq, plan, tma, x0, j, sm);
            if (x == kIcdfDead) return -1;
            if (threadIdx.x == 0) ph->tok = x;
        } else if (j.kind == kRadix) {
            for (int i = threadIdx.x; i < 256; i += kThreads) sm.bins[i] = 0;
            csync();
            RadixFn<E> fn;
            fn.bins = sm.bins;
            fn.round = j.aux2 & 0xff;
            fn.prefix = j.hint;
            if (!consume_row<E>(P, seq, plan, tma, x0, fn)) return -1;
            const float wv = block_max_nan(fn.vmx, sm.wm);
            csync();
            int* ob = reinterpret_cast<int*>(pk);
            for (int i = threadIdx.x; i < 256; i += kThreads) ob[i] = sm.bins[i];
            if (threadIdx.x == 0) {
                ph->flags = bad_max(wv) ? kPfBad : 0u;
                ph->vmax = wv;
            }
            nkeys = 128;   // 256 int bins = 1024 bytes
        }
        return static_cast<int>(sizeof(PartHdr)) + ((nkeys * 8 + 15) & ~15);
    }

    __device__ static Job combine(const Args& A, const Geo& G, const Job& j, const unsigned char* parts, Smem& sm) {
        switch (j.kind) {
            case kTk: return combine_topk<E>(A, G, j, parts, sm);
            case kSe: return combine_se<E>(A, G, j, parts, sm);
            case kResid: return combine_resid(A, G, j, parts);
            case kRescan: return combine_rescan<E>(A, j, parts, G.part_bytes, sm.last_hint);
            default: return combine_radix(A, G, j, parts);
        }
    }
};

template <class E, bool kTopk>
__global__ void __launch_bounds__(kBlockThreads, 1) chain_kernel(const ChainArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    Engine<ChainOp<E, kTopk>>::run(A, A.E.W, make_geo(A.E), smem);
}

template <class E, bool kTopk>
static const void* chain_fn() { return reinterpret_cast<const void*>(&chain_kernel<E, kTopk>); }

#ifdef SPEC_TEST_HOOKS
// test builds only: make the chain kernel's first posted job go missing
extern "C" int spec_test_drop_first_post(int on) {
    return static_cast<int>(cudaMemcpyToSymbol(g_test_drop_post, &on, sizeof(int)));
}
#endif

const void* chain_kernel_ptr(int ldt, bool topk) {
    if (ldt == 0) return topk ? chain_fn<F32, true>() : chain_fn<F32, false>();
    return topk ? chain_fn<BF16, true>() : chain_fn<BF16, false>();
}

size_t chain_smem(int C, int own, int part_bytes, int stages, int chunk) {
    // the same layout for every instantiation
    return Engine<ChainOp<F32, true>>::smem_bytes(C, own, part_bytes, stages, chunk);
}

int chain_part_bytes(int top_k, int cap_p) {
    const int keys = top_k > 0 ? (cap_p > 128 ? cap_p : 128) : 128;   // radix bins need 1 KiB
    return static_cast<int>(sizeof(PartHdr)) + keys * 8;
}

}  // namespace spec

#ifdef SPEC_TRACE
// development builds: install the chain kernels' event buffer and reset it
extern "C" int spec_trace_setup_chain(void* buf, unsigned cap) {
    unsigned z = 0;
    if (cudaMemcpyToSymbol(spec::g_trace, &buf, sizeof(buf)) != cudaSuccess) return 1;
    if (cudaMemcpyToSymbol(spec::g_trace_cap, &cap, sizeof(cap)) != cudaSuccess) return 1;
    return cudaMemcpyToSymbol(spec::g_trace_n, &z, sizeof(z)) != cudaSuccess;
}
extern "C" unsigned spec_trace_count_chain(void) {
    unsigned n = 0;
    cudaMemcpyFromSymbol(&n, spec::g_trace_n, sizeof(n));
    return n;
}
#endif
