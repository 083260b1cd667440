// spec_tree_build.cu -- DDTree best-first draft tree on the row-task engine.
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
// list (one task per depth: slices find their local top-M, the combine
// merges them).  The best-first enumeration then runs in the combining CTA:
// pop the best frontier entry, emit it, push its next sibling (same parent,
// next rank) and its first child (rank 0 of the next depth).  Every emitted
// entry's successors score no higher than it (q <= 1), so pops come out in
// non-increasing Q and the first `budget` pops are the best prefixes.  When a
// first child needs a depth whose list is not built yet, the enumeration
// saves its state to the workspace and pushes that depth's row task; depth
// rows past the last one the enumeration consults are never read.
#include "spec_chain.cuh"
#include "spec_select.cuh"

namespace spec {

constexpr int kBuildCap = kWarps * TopkSmem::kRegion;   // selected-list buffer (keys)

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

struct __align__(16) BuildSmem {
    TopkSmem tk;             // slice candidates; later the merged list and mask scratch
    PipeSmem pipe;
    int last;
    int lcnt;
    int oflow;
    uint64_t sh64[4];
    double red[kWarps];
    int ired[kWarps + 4];
    int hist[64];
    uint32_t scratch[kWarps + 2];
    EnumHdr eh;
    SliceHdrs hdrs;
};

// per-request extra scratch: [EnumHdr][lists L*M (tok,int) + (prob,float)][nodes N][pending 2N+2]
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
// dynamic shared memory beyond the ring and BuildSmem: scratch (depth lists,
// gathered keys and their ranks) + nodes + pending
constexpr int kBuildList = 2048;         // gathered keys in a combine
__host__ __device__ inline size_t build_lists_bytes(int N, int L) {
    return (static_cast<size_t>(L) * (N - 1) * 8 + 15) & ~static_cast<size_t>(15);
}
__host__ __device__ inline size_t build_scr_bytes(int N, int L) {
    return build_lists_bytes(N, L) + static_cast<size_t>(kBuildList) * 12;
}
static size_t build_enum_smem(int N, int L) {
    return build_scr_bytes(N, L) + static_cast<size_t>(3 * N + 2) * sizeof(Ent);
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

// Exact top-M (value desc, index asc) of one q row, single CTA, by
// bisection over composite keys; for rows whose slice candidate buffers
// overflowed (adversarial value order).  Writes the keys (unordered) to
// list[0..return).
__device__ int build_fallback(const float* qrow, int V, int M, uint64_t* list, int* ired, int* lcnt) {
    uint64_t lo = 0, hi = ~0ull;
    if (V > M) {
        // invariant: count(key >= lo) >= M; the range halves every step
        for (int it = 0; it < 66 && lo < hi; ++it) {
            const uint64_t d = hi - lo;
            const uint64_t mid = lo + (d >> 1) + (d & 1ull);
            int c = 0;
            for (int x = threadIdx.x; x < V; x += kThreads) c += ckey(qrow[x], x) >= mid;
            c = block_sum_i(c, ired);
            if (c >= M) lo = mid; else hi = mid - 1;
        }
    }
    if (threadIdx.x == 0) *lcnt = 0;
    csync();
    for (int x = threadIdx.x; x < V; x += kThreads) {
        const uint64_t key = ckey(qrow[x], x);
        if (key >= lo) {
            const int pos = atomicAdd(lcnt, 1);
            if (pos < M) list[pos] = key;
        }
    }
    csync();
    const int n = *lcnt;
    csync();
    return n < M ? n : M;
}

// Write the final tree of request b from shared memory (all threads).
__device__ void build_finalize(const BuildArgs& A, BuildSmem& sh, const Ent* nodes, const int* ltok,
                               int b, int count, int st) {
    const int N = A.N, M = A.M;
    const int W = (N + 63) / 64;
    int* tk = A.token + static_cast<long long>(b) * N;
    int* pr = A.parent + static_cast<long long>(b) * N;
    int* dp = A.depth + static_cast<long long>(b) * N;
    double* sc = A.score + static_cast<long long>(b) * N;
    for (int n = threadIdx.x; n < N; n += kThreads) {
        if (n < count) {
            const Ent& e = nodes[n];
            tk[n] = n == 0 ? -1 : ltok[(e.depth - 1) * M + e.rank];
            pr[n] = e.parent;
            dp[n] = e.depth;
            sc[n] = e.Q;
        } else {
            tk[n] = -1; pr[n] = -1; dp[n] = -1; sc[n] = 0.0;
        }
    }
    // ancestor masks: mask[n] = mask[parent[n]] | bit n, parents first
    unsigned long long* mk = A.anc_mask + static_cast<long long>(b) * N * W;
    unsigned long long* sm = reinterpret_cast<unsigned long long*>(sh.tk.cand);   // N*W <= 1024 words
    if (threadIdx.x == 0) {
        for (int n = 0; n < N; ++n) {
            for (int w = 0; w < W; ++w) {
                unsigned long long v = 0;
                if (n < count && nodes[n].parent >= 0) v = sm[nodes[n].parent * W + w];
                if (n < count && w == n / 64) v |= 1ull << (n % 64);
                sm[n * W + w] = v;
            }
        }
    }
    csync();
    for (int i = threadIdx.x; i < N * W; i += kThreads) mk[i] = sm[i];
    if (threadIdx.x == 0) {
        A.num_nodes[b] = count;
        A.status[b] = st;
    }
    csync();
    if (threadIdx.x == 0) finish_request(A.W);
}

__global__ void __launch_bounds__(kBlockThreads, 2) build_kernel(const BuildArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    auto& sh = *reinterpret_cast<BuildSmem*>(smem + kStages * kChunkBytes);
    unsigned char* scr = smem + kStages * kChunkBytes + sizeof(BuildSmem);
    Ent* nodes = reinterpret_cast<Ent*>(scr + build_scr_bytes(A.N, A.L));
    Ent* pend = nodes + A.N;
    const Pipe P = pipe_init(smem, sh.pipe);
    const int N = A.N, M = A.M, L = A.L;
    const bool tma = A.tma_q != 0;
    auto trivial_of = [&](const Task& t) { return t.kind < 0 && (N <= 1 || L <= 0); };
    auto plan = [&](const Task& t, int slice) {
        if (trivial_of(t)) return plan_none();
        const int x0 = slice * A.SL, x1 = min(A.V, x0 + A.SL);
        const float* qrow = A.q + static_cast<long long>(t.b) * A.q_bs + static_cast<long long>(t.row) * A.q_rs;
        return plan_single(qrow, 4, x0, x1);
    };
    if (threadIdx.x >= kThreads) {
        if (threadIdx.x == kThreads)
            producer_loop(A.W, A.B, A.S, P, tma, [](Claimed&) {},
                          [&](const Claimed& c) { return plan(c.task, c.slice); });
        return;
    }
    uint32_t seq = 0;
    for (uint32_t u = 0;; ++u) {
        const Claimed cl = next_unit(P, u);
        if (!cl.ok) break;
        const Task t = cl.task;
        const int s = cl.slice;
        const int b = t.b;
        const bool initial = t.kind < 0;
        const int d = t.row + 1;                 // depth of this row
        const bool trivial = trivial_of(t);
        PartHdr* ph = part_hdr(A.W, b, s, A.S);
        uint64_t* pk = part_keys(A.W, b, s, A.S);
        if (!trivial) {
            const int x0 = s * A.SL;
            TopkHistFn<F32, false> fn;
            fn.init(&sh.tk, M, 0u);
            if (!consume_row<F32>(P, seq, plan(t, s), tma, x0, fn)) break;
            uint64_t F;
            uint32_t oflow, bad;
            int n = fn.finish(F, oflow, bad);
            uint64_t* list = sh.tk.cand;
            if (n > A.cap_p && !bad) {
                // the slice's exact top-M (value desc, index asc); its M-th key is the filter
                uint64_t* dst = reinterpret_cast<uint64_t*>(scr);
                int* rank = reinterpret_cast<int*>(scr + static_cast<size_t>(A.cap_p) * 8);
                uint64_t kth;
                bool of2;
                n = select_to(list, n, M, false, rank, dst, A.cap_p, kth, of2, sh.sh64, sh.ired);
                F = kth;
                list = dst;
            }
            if (bad) n = 0;
            csync();
            for (int i = threadIdx.x; i < n; i += kThreads) __stcg(pk + i, list[i]);
            if (threadIdx.x == 0) {
                ph->flags = (bad ? kPfBad : 0u) | (oflow ? kPfOverflow : 0u);
                ph->cnt = n;
                ph->kth = F;
            }
        }
        if (!arrive(A.W, b, A.S, &sh.last)) continue;

        // ---- combine: merge the slice lists into depth d's sorted top-M ----
        unsigned char* ex = A.W.extra + static_cast<size_t>(b) * A.W.extra_stride;
        EnumHdr* gh = reinterpret_cast<EnumHdr*>(ex);
        int* gl = reinterpret_cast<int*>(ex + build_lists_off());        // [L][M] (tok, prob bits)
        Ent* gnodes = reinterpret_cast<Ent*>(ex + build_nodes_off(N, L));
        Ent* gpend = reinterpret_cast<Ent*>(ex + build_pend_off(N, L));
        // depth lists at the front of the ring: tokens [L*M] then probabilities [L*M]
        const int LM = L * M;
        int* ltok = reinterpret_cast<int*>(scr);
        float* lprob = reinterpret_cast<float*>(scr + static_cast<size_t>(LM) * 4);
        if (initial) {
            if (threadIdx.x == 0) {
                EnumHdr h{};
                h.count = 1; h.npend = 0; h.want = 0; h.avail = 0; h.status = 0;
                sh.eh = h;
            }
        } else {
            for (int i = threadIdx.x; i < static_cast<int>(sizeof(EnumHdr) / 4); i += kThreads)
                reinterpret_cast<int*>(&sh.eh)[i] = __ldcg(reinterpret_cast<const int*>(gh) + i);
        }
        csync();
        EnumHdr& eh = sh.eh;
        if (initial) {
            if (threadIdx.x == 0) {
                Ent root{};
                root.Q = 1.0; root.depth = 0; root.parent = -1; root.rank = -1;
                nodes[0] = root;
            }
        } else {
            const int nc = eh.count, np = eh.npend;
            for (int i = threadIdx.x; i < nc * 5; i += kThreads)
                reinterpret_cast<unsigned long long*>(nodes)[i] = __ldcg(reinterpret_cast<const unsigned long long*>(gnodes) + i);
            for (int i = threadIdx.x; i < np * 5; i += kThreads)
                reinterpret_cast<unsigned long long*>(pend)[i] = __ldcg(reinterpret_cast<const unsigned long long*>(gpend) + i);
            for (int i = threadIdx.x; i < eh.avail * M; i += kThreads) {
                ltok[i] = __ldcg(gl + 2 * i);
                lprob[i] = __int_as_float(__ldcg(gl + 2 * i + 1));
            }
        }
        csync();
        if (!trivial) {
            load_hdrs(A.W, b, A.S, sh.hdrs);
            uint32_t flags = 0;
            uint64_t theta = 0;
            for (int j = 0; j < A.S; ++j) {
                flags |= sh.hdrs.flags[j];
                theta = sh.hdrs.kth[j] > theta ? sh.hdrs.kth[j] : theta;
            }
            // gathered keys and their ranks in the rest of the ring
            uint64_t* list = reinterpret_cast<uint64_t*>(scr + build_lists_bytes(N, L));
            const int kList = kBuildList;
            int* rank = reinterpret_cast<int*>(list + kList);
            int n = 0;
            if (flags & kPfBad) {
                n = 0;
            } else if (flags & kPfOverflow) {
                const float* qrow = A.q + static_cast<long long>(b) * A.q_bs + static_cast<long long>(d - 1) * A.q_rs;
                n = build_fallback(qrow, A.V, M, list, sh.ired, &sh.lcnt);
            } else {
                // every slice key at or above the largest slice filter, then the top M
                gather_keys(A.W, b, A.S, sh.hdrs, [&](uint64_t key) { return key >= theta; }, list, kList,
                            &sh.lcnt, &sh.oflow);
                n = min(sh.lcnt, kList);
            }
            uint64_t kth;
            bool of;
            const int keep = (flags & kPfBad) ? 0
                             : select_to(list, n, M, false, rank, sh.tk.cand, kBuildCap, kth, of, sh.sh64, sh.ired);
            csync();
            for (int i = threadIdx.x; i < keep; i += kThreads) {
                const uint64_t key = sh.tk.cand[i];
                ltok[(d - 1) * M + i] = ckey_idx(key);
                lprob[(d - 1) * M + i] = ckey_val(key);
                __stcg(gl + 2 * ((d - 1) * M + i), ckey_idx(key));
                __stcg(gl + 2 * ((d - 1) * M + i) + 1, __float_as_int(ckey_val(key)));
            }
            if (threadIdx.x == 0) {
                eh.len[d] = keep;
                eh.avail = d;
                if (flags & kPfBad) eh.status |= 1;
            }
            csync();
        }
        // ---- best-first enumeration (thread 0), resumable ----
        if (threadIdx.x == 0) {
            int count = eh.count, np = eh.npend, want = eh.want;
            int need = 0;
            while (count < N) {
                if (want >= 0) {
                    const int dd = nodes[want].depth + 1;
                    if (dd <= L) {
                        if (dd > eh.avail) { need = dd; break; }
                        if (eh.len[dd] > 0) {
                            Ent c = nodes[want];
                            c.depth = dd; c.parent = want; c.rank = 0;
                            path_set(c, dd, 0);
                            c.Q = nodes[want].Q * static_cast<double>(lprob[(dd - 1) * M + 0]);
                            pend[np++] = c;
                        }
                    }
                    want = -1;
                }
                if (np == 0) break;
                int best = 0;
                for (int j = 1; j < np; ++j)
                    if (ent_before(pend[j], pend[best])) best = j;
                const Ent c = pend[best];
                pend[best] = pend[--np];
                const int nid = count++;
                nodes[nid] = c;
                if (c.rank + 1 < eh.len[c.depth]) {
                    Ent s2 = c;
                    s2.rank = c.rank + 1;
                    path_set(s2, c.depth, c.rank + 1);
                    s2.Q = nodes[c.parent].Q * static_cast<double>(lprob[(c.depth - 1) * M + c.rank + 1]);
                    pend[np++] = s2;
                }
                want = nid;
            }
            eh.count = count; eh.npend = np; eh.want = want;
            sh.ired[0] = need;
        }
        csync();
        const int need = sh.ired[0];
        if (need == 0) {
            build_finalize(A, sh, nodes, ltok, b, eh.count, eh.status);
        } else {
            // save the state and ask for depth `need`
            const int nc = eh.count, np = eh.npend;
            for (int i = threadIdx.x; i < nc * 5; i += kThreads)
                __stcg(reinterpret_cast<unsigned long long*>(gnodes) + i, reinterpret_cast<const unsigned long long*>(nodes)[i]);
            for (int i = threadIdx.x; i < np * 5; i += kThreads)
                __stcg(reinterpret_cast<unsigned long long*>(gpend) + i, reinterpret_cast<const unsigned long long*>(pend)[i]);
            for (int i = threadIdx.x; i < static_cast<int>(sizeof(EnumHdr) / 4); i += kThreads)
                __stcg(reinterpret_cast<int*>(gh) + i, reinterpret_cast<const int*>(&eh)[i]);
            csync();
            if (threadIdx.x == 0) {
                Task nt;
                nt.b = b; nt.row = need - 1; nt.kind = 0; nt.aux = 0;
                push_task(A.W, nt);
            }
        }
        csync();
    }
}

// largest slice count whose candidate lists fit the combine's gather buffer
int build_max_slices(int N, int L) {
    (void)L;
    const int M = N - 1;
    const int s = M > 0 ? kBuildList / M : kMaxSlices;
    return s < 1 ? 1 : (s > kMaxSlices ? kMaxSlices : s);
}

static size_t build_smem(int N, int L) { return kStages * kChunkBytes + sizeof(BuildSmem) + build_enum_smem(N, L); }

int build_occupancy(int N, int L) {
    const int smem = static_cast<int>(build_smem(N, L));
    int n = 0;
    cudaFuncSetAttribute(build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, build_kernel, kBlockThreads, smem);
    return n;
}

cudaError_t build_run(const BuildArgs& A, int grid, cudaStream_t st) {
    const size_t smem = build_smem(A.N, A.L);
    cudaError_t e = cudaFuncSetAttribute(build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    build_kernel<<<grid, kBlockThreads, smem, st>>>(A);
    return cudaGetLastError();
}

}  // namespace spec
