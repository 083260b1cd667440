// spec_tree_build.cu -- DDTree best-first draft tree on the cluster engine.
//
// [SD-survey] = "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
// (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash, DDTree and
// DSpark), chzhyang.github.io, §5 "DDTree": a prefix u is scored by the
// factorised proxy Q(u) = prod_{i=1}^{|u|} q_i(u_i); a best-first heap picks
// prefixes under a node budget; node position id = depth; a node sees only
// itself and its ancestors.
//
// Depth d contributes at most M = budget-1 nodes, all among the M most
// probable tokens of q_d, so each depth row is reduced to its sorted top-M
// list: one job per depth, in which every CTA of the cluster finds its
// slice's top-M composite keys and the slot's leader merges them.  The
// best-first enumeration then runs on the leader's combiner warp: each pop is
// a warp-wide arg-max over the frontier; the popped entry is emitted and its
// next sibling (same parent, next rank) and first child (rank 0 of the next
// depth) join the frontier.  Every emitted entry's successors score no
// higher than it (q <= 1), so pops come out in non-increasing Q and the first
// `budget` pops are the best prefixes.  When a first child needs a depth
// whose list is not built yet, the enumeration saves its state to the
// workspace and posts that depth's row job; depth rows past the last one the
// enumeration consults are never read.
#include "spec_chain.cuh"
#include "spec_select.cuh"

namespace spec {

struct Ent {                 // a frontier entry or an emitted node
    double Q;
    unsigned long long ph, pl;   // rank path, one byte per depth, depth 1 in the top byte
    int depth, parent, rank, pad;
};
static_assert(sizeof(Ent) == 40, "Ent is 40 bytes");

struct EnumHdr {
    int count, npend, want, avail;
    int status, pad[3];
    int len[24];             // list length per depth (index 1..L)
};

constexpr int kBuildList = 2048;         // gathered keys in a combine (at most C * M)

struct BuildSmem {
    TopkSmem tk;             // consumers: slice candidates
    uint64_t sh64[4];
    int ired[kWarps + 4];
    int hist[64];
    uint32_t scratch[kWarps + 2];
    EnumHdr eh;              // combiner
    alignas(16) uint64_t list[kBuildList];   // combiner: gathered keys
};

// per-request workspace: [EnumHdr][lists L*M (tok, prob bits)][nodes N][pending 2N+2]
__host__ __device__ inline size_t build_lists_off() { return 128; }
__host__ __device__ inline size_t build_nodes_off(int N, int L) {
    return (build_lists_off() + static_cast<size_t>(L) * (N - 1) * 8 + 127) & ~static_cast<size_t>(127);
}
__host__ __device__ inline size_t build_pend_off(int N, int L) {
    return build_nodes_off(N, L) + static_cast<size_t>(N) * sizeof(Ent);
}
size_t build_extra_bytes(int N, int L) {
    return (build_pend_off(N, L) + static_cast<size_t>(2 * N + 2) * sizeof(Ent) + 127) & ~static_cast<size_t>(127);
}
// combiner shared memory after the partial areas: depth lists, nodes and pending
__host__ __device__ inline size_t enum_smem_bytes(int N, int L) {
    return ((static_cast<size_t>(L) * (N - 1) * 8 + 15) & ~static_cast<size_t>(15)) +
           static_cast<size_t>(3 * N + 2) * sizeof(Ent);
}

__device__ __forceinline__ bool ent_before(const Ent& a, const Ent& b) {
    if (a.Q != b.Q) return a.Q > b.Q;
    if (a.depth != b.depth) return a.depth < b.depth;
    if (a.ph != b.ph) return a.ph < b.ph;
    return a.pl < b.pl;
}
__device__ __forceinline__ void path_set(Ent& e, int d, int r) {
    const unsigned long long v = static_cast<unsigned long long>(r & 0xff);
    if (d <= 8) {
        const int sh = 8 * (8 - d);
        e.ph = (e.ph & ~(0xffull << sh)) | (v << sh);
    } else {
        const int sh = 8 * (16 - d);
        e.pl = (e.pl & ~(0xffull << sh)) | (v << sh);
    }
}

// the enumeration's shared-memory view (combiner warp): depth lists
// (tokens, probabilities), emitted nodes, frontier
struct EnumView {
    int* ltok;
    float* lprob;
    Ent* nodes;
    Ent* pend;
};
__device__ __forceinline__ EnumView enum_view(unsigned char* base, int N, int L) {
    EnumView v;
    const int LM = L * (N - 1);
    v.ltok = reinterpret_cast<int*>(base);
    v.lprob = reinterpret_cast<float*>(base + static_cast<size_t>(LM) * 4);
    v.nodes = reinterpret_cast<Ent*>(base + ((static_cast<size_t>(LM) * 8 + 15) & ~static_cast<size_t>(15)));
    v.pend = v.nodes + N;
    return v;
}

// Write the final tree of request b (combiner warp).
__device__ void build_finalize(const BuildArgs& A, const EnumView& ev, int b, int count, int st) {
    const int l = threadIdx.x & 31;
    const int N = A.N, M = A.M;
    const int W = (N + 63) / 64;
    int* tk = A.token + static_cast<long long>(b) * N;
    int* pr = A.parent + static_cast<long long>(b) * N;
    int* dp = A.depth + static_cast<long long>(b) * N;
    double* sc = A.score + static_cast<long long>(b) * N;
    unsigned long long* mk = A.anc_mask + static_cast<long long>(b) * N * W;
    for (int n = l; n < N; n += 32) {
        if (n < count) {
            const Ent& e = ev.nodes[n];
            tk[n] = n == 0 ? -1 : ev.ltok[(e.depth - 1) * M + e.rank];
            pr[n] = e.parent;
            dp[n] = e.depth;
            sc[n] = e.Q;
        } else {
            tk[n] = -1; pr[n] = -1; dp[n] = -1; sc[n] = 0.0;
        }
        // ancestor mask: the node itself and every ancestor (parents precede
        // children, so the walk up ends at the root); W <= 4 words (N <= 256)
        unsigned long long mw[4] = {0ull, 0ull, 0ull, 0ull};
        if (n < count) {
            int m = n;
            for (int guard = 0; m >= 0 && guard <= N; ++guard) {
                mw[m / 64] |= 1ull << (m % 64);
                m = ev.nodes[m].parent;
            }
        }
        for (int w = 0; w < W; ++w) mk[static_cast<long long>(n) * W + w] = mw[w];
    }
    if (l == 0) {
        A.num_nodes[b] = count;
        A.status[b] = st;
    }
    __syncwarp();
}

// warp-wide pop of the best frontier entry: its index in every lane
__device__ __forceinline__ int best_pending_w(const Ent* pend, int np) {
    const int l = threadIdx.x & 31;
    int best = -1;
    for (int j = l; j < np; j += 32)
        if (best < 0 || ent_before(pend[j], pend[best])) best = j;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const int other = __shfl_xor_sync(0xffffffffu, best, o);
        if (other >= 0 && (best < 0 || ent_before(pend[other], pend[best]) ||
                           (!ent_before(pend[best], pend[other]) && other < best)))
            best = other;
    }
    return best;
}

// The best-first enumeration from the saved state in `eh` / `ev` (combiner
// warp).  Returns the depth whose list it needs next, or 0 when the tree is
// complete.
__device__ int enumerate_w(const BuildArgs& A, EnumHdr& eh, const EnumView& ev) {
    const int l = threadIdx.x & 31;
    const int N = A.N, M = A.M, L = A.L;
    int count = eh.count, np = eh.npend, want = eh.want;
    int need = 0;
    while (count < N) {
        if (want >= 0) {
            const int dd = ev.nodes[want].depth + 1;
            if (dd <= L) {
                if (dd > eh.avail) { need = dd; break; }
                if (eh.len[dd] > 0) {
                    if (l == 0) {
                        Ent c = ev.nodes[want];
                        c.depth = dd; c.parent = want; c.rank = 0;
                        path_set(c, dd, 0);
                        c.Q = ev.nodes[want].Q * static_cast<double>(ev.lprob[(dd - 1) * M + 0]);
                        ev.pend[np] = c;
                    }
                    ++np;
                    __syncwarp();
                }
            }
            want = -1;
        }
        if (np == 0) break;
        const int best = best_pending_w(ev.pend, np);
        const Ent c = ev.pend[best];
        __syncwarp();
        if (l == 0) {
            ev.pend[best] = ev.pend[np - 1];
            ev.nodes[count] = c;
        }
        --np;
        const int nid = count++;
        if (c.rank + 1 < eh.len[c.depth]) {
            if (l == 0) {
                Ent s2 = c;
                s2.rank = c.rank + 1;
                path_set(s2, c.depth, c.rank + 1);
                s2.Q = ev.nodes[c.parent].Q * static_cast<double>(ev.lprob[(c.depth - 1) * M + c.rank + 1]);
                ev.pend[np] = s2;
            }
            ++np;
        }
        __syncwarp();
        want = nid;
    }
    if (l == 0) { eh.count = count; eh.npend = np; eh.want = want; }
    __syncwarp();
    return need;
}

// save / load the enumeration state of request b (combiner warp; the
// workspace lines bypass L1)
__device__ void enum_save(const BuildArgs& A, int b, const EnumHdr& eh, const EnumView& ev, int first_list) {
    const int l = threadIdx.x & 31;
    const int N = A.N, M = A.M, L = A.L;
    unsigned char* ex = A.E.W.extra + static_cast<size_t>(b) * A.E.W.extra_stride;
    int* gl = reinterpret_cast<int*>(ex + build_lists_off());
    const int nc = eh.count, np = eh.npend;
    for (int i = l; i < nc * 5; i += 32)
        __stcg(reinterpret_cast<unsigned long long*>(ex + build_nodes_off(N, L)) + i,
               reinterpret_cast<const unsigned long long*>(ev.nodes)[i]);
    for (int i = l; i < np * 5; i += 32)
        __stcg(reinterpret_cast<unsigned long long*>(ex + build_pend_off(N, L)) + i,
               reinterpret_cast<const unsigned long long*>(ev.pend)[i]);
    for (int i = first_list * M + l; i < eh.avail * M; i += 32) {
        __stcg(gl + 2 * i, ev.ltok[i]);
        __stcg(gl + 2 * i + 1, __float_as_int(ev.lprob[i]));
    }
    for (int i = l; i < static_cast<int>(sizeof(EnumHdr) / 4); i += 32)
        __stcg(reinterpret_cast<int*>(ex) + i, reinterpret_cast<const int*>(&eh)[i]);
    __syncwarp();
}
__device__ void enum_load(const BuildArgs& A, int b, EnumHdr& eh, const EnumView& ev) {
    const int l = threadIdx.x & 31;
    const int N = A.N, M = A.M, L = A.L;
    const unsigned char* ex = A.E.W.extra + static_cast<size_t>(b) * A.E.W.extra_stride;
    const int* gl = reinterpret_cast<const int*>(ex + build_lists_off());
    for (int i = l; i < static_cast<int>(sizeof(EnumHdr) / 4); i += 32)
        reinterpret_cast<int*>(&eh)[i] = __ldcg(reinterpret_cast<const int*>(ex) + i);
    __syncwarp();
    const int nc = eh.count, np = eh.npend;
    for (int i = l; i < nc * 5; i += 32)
        reinterpret_cast<unsigned long long*>(ev.nodes)[i] =
            __ldcg(reinterpret_cast<const unsigned long long*>(ex + build_nodes_off(N, L)) + i);
    for (int i = l; i < np * 5; i += 32)
        reinterpret_cast<unsigned long long*>(ev.pend)[i] =
            __ldcg(reinterpret_cast<const unsigned long long*>(ex + build_pend_off(N, L)) + i);
    for (int i = l; i < eh.avail * M; i += 32) {
        ev.ltok[i] = __ldcg(gl + 2 * i);
        ev.lprob[i] = __int_as_float(__ldcg(gl + 2 * i + 1));
    }
    __syncwarp();
}

// The row's M largest composite keys (value desc, index asc) from the
// slices' reports, on the combiner warp: every key at or above the largest
// slice filter, cut to exactly M (composite keys are unique).  A slice
// overflow, or more keys than the list holds, re-derives them from the row
// itself.  `flags`, `theta` (the largest slice filter) and `cnt` (lane r:
// slice r's key count) come from the headers.  Keys, unordered, to
// list[0..return); 0 for a bad row.
__device__ int merge_topm_w(const unsigned char* parts, int pb, int C, int M, uint32_t flags, uint64_t theta, int cnt,
                            const float* qrow, int V, uint64_t* list);

struct BuildOp {
    using Args = BuildArgs;
    using Smem = BuildSmem;

    __device__ static int batch(const Args& A) { return A.B; }
    __device__ static bool tma(const Args& A) { return A.tma_q != 0; }
    __device__ static void init_smem(const Args&, const Geo&, Smem& sm) {
        if (threadIdx.x == 0) topk_smem_init(sm.tk);
    }
    // the combiner's enumeration scratch sits after the ring
    __device__ static EnumView view(const Args& A, const Geo& G) {
        extern __shared__ __align__(128) unsigned char smem[];
        const size_t off = Engine<BuildOp>::smem_bytes(G.C, G.own, G.part_bytes, G.stages, G.chunk);
        return enum_view(smem + ((off + 15) & ~static_cast<size_t>(15)), A.N, A.L);
    }
    __device__ static Job first(const Args& A, const Geo& G, int b, Smem& sm) {
        const int l = threadIdx.x & 31;
        const EnumView ev = view(A, G);
        EnumHdr& eh = sm.eh;
        if (l == 0) {
            EnumHdr h{};
            h.count = 1; h.npend = 0; h.want = 0; h.avail = 0; h.status = 0;
            eh = h;
            Ent root{};
            root.Q = 1.0; root.depth = 0; root.parent = -1; root.rank = -1;
            ev.nodes[0] = root;
        }
        __syncwarp();
        if (A.N <= 1 || A.L <= 0) {
            build_finalize(A, ev, b, 1, 0);
            return job_done();
        }
        enum_save(A, b, eh, ev, 0);
        return make_job(b, 0, 0, 0);   // depth 1's row
    }
    __device__ static StreamPlan plan(const Args& A, const Geo& G, const Job& j) {
        const float* qrow = A.q + static_cast<long long>(j.b) * A.q_bs + static_cast<long long>(j.row) * A.q_rs;
        return plan_single(qrow, 4, slice_x0(G, G.rank), slice_x1(G, G.rank, A.V), G.chunk);
    }
    // consumers: this slice's top-M composite keys (value desc, index asc)
    __device__ static int consume(const Args& A, const Geo& G, const Pipe& P, uint32_t& seq, bool tma, const Job& j,
                                  Smem& sm, unsigned char* out) {
        PartHdr* ph = reinterpret_cast<PartHdr*>(out);
        uint64_t* pk = reinterpret_cast<uint64_t*>(ph + 1);
        const int M = A.M;
        TopkHistFn<F32, false> fn;
        fn.init(&sm.tk, M, 0u, seq + 1u);   // every consumer holds the same seq
        if (!consume_row<F32>(P, seq, plan(A, G, j), tma, slice_x0(G, G.rank), fn)) return -1;
        uint64_t F;
        uint32_t oflow, bad;
        float vm;
        int n = fn.finish(F, oflow, bad, vm);
        uint64_t* list = sm.tk.cand;
        if (n > A.cap_p && !bad && !oflow) {
            // the slice's exact M-th key: a certified value bound (repeated
            // until it stops rising), then the index bits within that value
            for (int it = 0; it < 8 && n > A.cap_p; ++it) {
                bool cert;
                const uint32_t F2 = hist_bound_list(list, n, M, hkey(F), sm.hist, sm.scratch, cert);
                if (!(cert && F2 > hkey(F))) break;
                n = compact_list(list, n, F2, sm.ired);
                F = static_cast<uint64_t>(F2) << 32;
            }
            if (n > A.cap_p) {
                const uint64_t kth = composite_bound(
                    [&](auto f) { for (int i = threadIdx.x; i < n; i += kThreads) f(list[i]); }, M, F, sm.ired);
                // keep the keys >= kth (order kept)
                int outn = 0;
                const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
                for (int i0 = 0; i0 < n; i0 += kThreads) {
                    const int i = i0 + threadIdx.x;
                    uint64_t key = 0;
                    bool p = false;
                    if (i < n) { key = list[i]; p = key >= kth; }
                    const uint32_t bal = __ballot_sync(0xffffffffu, p);
                    if (lane == 0) sm.ired[w] = __popc(bal);
                    csync();
                    int base = outn, tot = 0;
                    for (int q = 0; q < kWarps; ++q) {
                        if (q < w) base += sm.ired[q];
                        tot += sm.ired[q];
                    }
                    csync();
                    if (p) list[base + __popc(bal & ((1u << lane) - 1u))] = key;
                    outn += tot;
                    csync();
                }
                n = outn;
                F = kth;
                if (n > A.cap_p) oflow = 1;
            }
        }
        if (bad || oflow) n = 0;
        csync();
        for (int i = threadIdx.x; i < n; i += kThreads) pk[i] = list[i];
        if (threadIdx.x == 0) {
            ph->flags = (bad ? kPfBad : 0u) | (oflow ? kPfOverflow : 0u);
            ph->cnt = n;
            ph->kth = F;
        }
        return static_cast<int>(sizeof(PartHdr)) + ((n * 8 + 15) & ~15);
    }

    // Exact top-M (value desc, index asc) of one q row by bisection over
    // composite keys, on the combiner warp; for rows whose slice candidate
    // buffers overflowed (adversarial value order).  Keys (unordered) to
    // list[0..return).
    __device__ static int fallback(const float* qrow, int V, int M, uint64_t* list) {
        const int l = threadIdx.x & 31;
        uint64_t lo = 0, hi = ~0ull;
        if (V > M) {
            // invariant: count(key >= lo) >= M; the range halves every step
            for (int it = 0; it < 66 && lo < hi; ++it) {
                const uint64_t d = hi - lo;
                const uint64_t mid = lo + (d >> 1) + (d & 1ull);
                int c = 0;
                for (int x = l; x < V; x += 32) c += ckey(qrow[x], x) >= mid;
                c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(c)));
                if (c >= M) lo = mid; else hi = mid - 1;
            }
        }
        const uint32_t lt = (1u << l) - 1u;
        int out = 0;
        for (int x0 = 0; x0 < V; x0 += 32) {
            const int x = x0 + l;
            uint64_t key = 0;
            bool p = false;
            if (x < V) { key = ckey(qrow[x], x); p = key >= lo; }
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            if (p) {
                const int pos = out + __popc(bal & lt);
                if (pos < M) list[pos] = key;
            }
            out += __popc(bal);
        }
        __syncwarp();
        return out < M ? out : M;
    }

    __device__ static Job combine(const Args& A, const Geo& G, const Job& j, const unsigned char* parts, Smem& sm) {
        const int l = threadIdx.x & 31;
        const int M = A.M, C = G.C, pb = G.part_bytes;
        const int b = j.b;
        const int d = j.row + 1;
        const EnumView ev = view(A, G);
        EnumHdr& eh = sm.eh;
        enum_load(A, b, eh, ev);
        uint32_t flags = 0;
        uint64_t theta = 0;
        int cnt = 0;
        if (l < C) {
            const PartHdr* h = part_at(parts, pb, l);
            flags = h->flags; theta = h->kth; cnt = h->cnt;
        }
        flags = __reduce_or_sync(0xffffffffu, flags);
        theta = warp_max_u64(theta);
        const float* qrow = A.q + static_cast<long long>(b) * A.q_bs + static_cast<long long>(d - 1) * A.q_rs;
        uint64_t* list = sm.list;
        const int n = merge_topm_w(parts, pb, C, M, flags, theta, cnt, qrow, A.V, list);
        // the depth list in rank order (value desc, index asc)
        for (int i = l; i < n; i += 32) {
            const uint64_t key = list[i];
            int r = 0;
            for (int q = 0; q < n; ++q) r += list[q] > key;
            const int o = (d - 1) * M + r;
            ev.ltok[o] = ckey_idx(key);
            ev.lprob[o] = ckey_val(key);
        }
        if (l == 0) {
            eh.len[d] = n;
            eh.avail = d;
            if (flags & kPfBad) eh.status |= 1;
        }
        __syncwarp();
        const int need = enumerate_w(A, eh, ev);
        if (need == 0) {
            build_finalize(A, ev, b, eh.count, eh.status);
            return job_done();
        }
        enum_save(A, b, eh, ev, d - 1);
        return make_job(b, need - 1, 0, 0);
    }
};

__device__ int merge_topm_w(const unsigned char* parts, int pb, int C, int M, uint32_t flags, uint64_t theta, int cnt,
                            const float* qrow, int V, uint64_t* list) {
    const int l = threadIdx.x & 31;
    if (flags & kPfBad) return 0;
    if (flags & kPfOverflow) return BuildOp::fallback(qrow, V, M, list);
    const uint32_t lt = (1u << l) - 1u;
    int n = 0;
    for (int r = 0; r < C; ++r) {
        const int cr = __shfl_sync(0xffffffffu, cnt, r);
        const uint64_t* keys = reinterpret_cast<const uint64_t*>(part_at(parts, pb, r) + 1);
        for (int i0 = 0; i0 < cr; i0 += 32) {
            const int i = i0 + l;
            uint64_t key = 0;
            bool p = false;
            if (i < cr) { key = keys[i]; p = key >= theta; }
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            if (p) {
                const int pos = n + __popc(bal & lt);
                if (pos < kBuildList) list[pos] = key;
            }
            n += __popc(bal);
        }
    }
    __syncwarp();
    if (n > kBuildList) return BuildOp::fallback(qrow, V, M, list);
    if (n > M) {
        const uint64_t kth = kth_key_w(list, n, M);
        n = compact_key_w(list, n, kth);   // exactly M: composite keys are unique
    }
    return n;
}

// ---------------------------------------------------------------------------
// EAGLE-2 expansion rows ([SD-survey] §4 "EAGLE-2"): every frontier node's
// conditional draft row reduced to its K2 most probable tokens (probability
// descending, lower id first), one engine unit per (request, frontier slot),
// so that every row of the step streams in parallel.
// ---------------------------------------------------------------------------
size_t eagle_row_extra_bytes(int K2) { return sizeof(EagleRowHdr) + static_cast<size_t>(K2 > 0 ? K2 : 1) * 8; }

struct EagleOp {
    using Args = EagleArgs;
    using Smem = BuildSmem;

    __device__ static int batch(const Args& A) { return A.base.B * A.F; }
    __device__ static bool tma(const Args& A) { return A.base.tma_q != 0; }
    __device__ static void init_smem(const Args&, const Geo&, Smem& sm) {
        if (threadIdx.x == 0) topk_smem_init(sm.tk);
    }
    __device__ static EagleRowHdr* row_hdr(const Args& A, int u) {
        return reinterpret_cast<EagleRowHdr*>(A.base.E.W.extra + static_cast<size_t>(u) * A.base.E.W.extra_stride);
    }
    __device__ static Job first(const Args& A, const Geo&, int u, Smem&) {
        const int b = u / A.F, f = u - b * A.F;
        int nf = A.num_front_in[b];
        nf = nf < 0 ? 0 : (nf > A.F ? A.F : nf);
        int n = 0;
        if (f >= nf) {
            n = -1;
        } else {
            // node ids below the (valid) generated count
            const int g = A.num_gen[b];
            const int g0 = g < 1 ? 0 : (g > A.G ? A.G : g);
            const int id = A.front_in[static_cast<long long>(b) * A.F + f];
            if (id < 0 || id >= g0) n = -2;
        }
        if (n < 0) {
            if ((threadIdx.x & 31) == 0) {
                EagleRowHdr* h = row_hdr(A, u);
                h->n = n;
                h->bad = 0;
            }
            __syncwarp();
            return job_done();
        }
        return make_job(b, f, 0, 0);
    }
    __device__ static StreamPlan plan(const Args& A, const Geo& G, const Job& j) { return BuildOp::plan(A.base, G, j); }
    __device__ static int consume(const Args& A, const Geo& G, const Pipe& P, uint32_t& seq, bool tma, const Job& j,
                                  Smem& sm, unsigned char* out) {
        return BuildOp::consume(A.base, G, P, seq, tma, j, sm, out);
    }
    __device__ static Job combine(const Args& A, const Geo& G, const Job& j, const unsigned char* parts, Smem& sm) {
        const int l = threadIdx.x & 31;
        const int M = A.base.M, C = G.C, pb = G.part_bytes;
        uint32_t flags = 0;
        uint64_t theta = 0;
        int cnt = 0;
        if (l < C) {
            const PartHdr* h = part_at(parts, pb, l);
            flags = h->flags; theta = h->kth; cnt = h->cnt;
        }
        flags = __reduce_or_sync(0xffffffffu, flags);
        theta = warp_max_u64(theta);
        const float* qrow = A.base.q + static_cast<long long>(j.b) * A.base.q_bs +
                            static_cast<long long>(j.row) * A.base.q_rs;
        const int n = merge_topm_w(parts, pb, C, M, flags, theta, cnt, qrow, A.base.V, sm.list);
        const int u = j.b * A.F + j.row;
        EagleRowHdr* h = row_hdr(A, u);
        int* tok = reinterpret_cast<int*>(h + 1);
        float* prob = reinterpret_cast<float*>(tok + M);
        for (int i = l; i < n; i += 32) {
            const uint64_t key = sm.list[i];
            int r = 0;
            for (int q = 0; q < n; ++q) r += sm.list[q] > key;
            tok[r] = ckey_idx(key);
            prob[r] = ckey_val(key);
        }
        if (l == 0) {
            h->n = n;
            h->bad = (flags & kPfBad) ? 1 : 0;
        }
        __syncwarp();
        return job_done();
    }
};

__global__ void __launch_bounds__(kBlockThreads, 1) eagle_rows_kernel(const EagleArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    Engine<EagleOp>::run(A, A.base.E.W, make_geo(A.base.E), smem);
}
const void* eagle_rows_kernel_ptr() { return reinterpret_cast<const void*>(&eagle_rows_kernel); }
size_t eagle_rows_smem(int C, int own, int part_bytes, int stages, int chunk) {
    return Engine<EagleOp>::smem_bytes(C, own, part_bytes, stages, chunk);
}

__global__ void __launch_bounds__(kBlockThreads, 1) build_kernel(const BuildArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    Engine<BuildOp>::run(A, A.E.W, make_geo(A.E), smem);
}

const void* build_kernel_ptr() { return reinterpret_cast<const void*>(&build_kernel); }

size_t build_smem(int C, int own, int part_bytes, int stages, int chunk, int N, int L) {
    return ((Engine<BuildOp>::smem_bytes(C, own, part_bytes, stages, chunk) + 15) & ~static_cast<size_t>(15)) +
           enum_smem_bytes(N, L);
}
int build_part_bytes(int M) { return static_cast<int>(sizeof(PartHdr)) + ((M > 0 ? M : 1) * 8 + 15) / 16 * 16; }

}  // namespace spec
