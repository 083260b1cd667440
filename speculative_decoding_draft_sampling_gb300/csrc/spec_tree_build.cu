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
    TopkSmem tk;             // slice candidates (consumers)
    PipeSmem pipe;
    uint64_t sh64[4];
    double red[kWarps];
    int ired[kWarps + 4];
    int hist[64];
    uint32_t scratch[kWarps + 2];
    EnumHdr eh;              // combiner
    SliceHdrs hdrs;          // combiner
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
// dynamic shared memory beyond the ring and BuildSmem, all the combiner's:
// depth lists, gathered keys, ancestor-mask scratch, then nodes + pending
constexpr int kBuildList = 2048;         // gathered keys in a combine
__host__ __device__ inline size_t build_lists_bytes(int N, int L) {
    return (static_cast<size_t>(L) * (N - 1) * 8 + 15) & ~static_cast<size_t>(15);
}
__host__ __device__ inline size_t build_mask_off(int N, int L) {
    return build_lists_bytes(N, L) + static_cast<size_t>(kBuildList) * 8;
}
__host__ __device__ inline size_t build_scr_bytes(int N, int L) {
    return build_mask_off(N, L) + static_cast<size_t>(N) * ((N + 63) / 64) * 8;
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

// Exact top-M (value desc, index asc) of one q row by bisection over
// composite keys, on the combiner warp; for rows whose slice candidate
// buffers overflowed (adversarial value order).  Writes the keys
// (unordered) to list[0..return).
__device__ int build_fallback(const float* qrow, int V, int M, uint64_t* list) {
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

// Write the final tree of request b from shared memory (combiner warp).
__device__ void build_finalize(const BuildArgs& A, unsigned long long* msk, const Ent* nodes, const int* ltok,
                               int b, int count, int st) {
    const int l = threadIdx.x & 31;
    const int N = A.N, M = A.M;
    const int W = (N + 63) / 64;
    int* tk = A.token + static_cast<long long>(b) * N;
    int* pr = A.parent + static_cast<long long>(b) * N;
    int* dp = A.depth + static_cast<long long>(b) * N;
    double* sc = A.score + static_cast<long long>(b) * N;
    for (int n = l; n < N; n += 32) {
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
    if (l == 0) {
        for (int n = 0; n < N; ++n) {
            for (int w = 0; w < W; ++w) {
                unsigned long long v = 0;
                if (n < count && nodes[n].parent >= 0) v = msk[nodes[n].parent * W + w];
                if (n < count && w == n / 64) v |= 1ull << (n % 64);
                msk[n * W + w] = v;
            }
        }
    }
    __syncwarp();
    for (int i = l; i < N * W; i += 32) mk[i] = msk[i];
    if (l == 0) {
        A.num_nodes[b] = count;
        A.status[b] = st;
    }
    __syncwarp();
    if (l == 0) finish_request(A.W);
}

// The combine of one depth row (combiner warp): merge the slice lists into
// the depth's sorted top-M, then resume the best-first enumeration.
__device__ void build_combine(const BuildArgs& A, BuildSmem& sh, unsigned char* scr, Ent* nodes, Ent* pend,
                              const Job& job, uint32_t done, uint32_t base) {
    const int l = threadIdx.x & 31;
    const int N = A.N, M = A.M, L = A.L;
    const int b = job.task.b;
    const bool initial = job.task.kind < 0;
    const int d = job.task.row + 1;
    const bool trivial = job.kind != 0;
    unsigned char* ex = A.W.extra + static_cast<size_t>(b) * A.W.extra_stride;
    EnumHdr* gh = reinterpret_cast<EnumHdr*>(ex);
    int* gl = reinterpret_cast<int*>(ex + build_lists_off());        // [L][M] (tok, prob bits)
    Ent* gnodes = reinterpret_cast<Ent*>(ex + build_nodes_off(N, L));
    Ent* gpend = reinterpret_cast<Ent*>(ex + build_pend_off(N, L));
    const int LM = L * M;
    int* ltok = reinterpret_cast<int*>(scr);
    float* lprob = reinterpret_cast<float*>(scr + static_cast<size_t>(LM) * 4);
    uint64_t* list = reinterpret_cast<uint64_t*>(scr + build_lists_bytes(N, L));
    unsigned long long* msk = reinterpret_cast<unsigned long long*>(scr + build_mask_off(N, L));
    EnumHdr& eh = sh.eh;
    if (initial) {
        if (l == 0) {
            EnumHdr h{};
            h.count = 1; h.npend = 0; h.want = 0; h.avail = 0; h.status = 0;
            eh = h;
            Ent root{};
            root.Q = 1.0; root.depth = 0; root.parent = -1; root.rank = -1;
            nodes[0] = root;
        }
    } else {
        for (int i = l; i < static_cast<int>(sizeof(EnumHdr) / 4); i += 32)
            reinterpret_cast<int*>(&eh)[i] = __ldcg(reinterpret_cast<const int*>(gh) + i);
        __syncwarp();
        const int nc = eh.count, np = eh.npend;
        for (int i = l; i < nc * 5; i += 32)
            reinterpret_cast<unsigned long long*>(nodes)[i] = __ldcg(reinterpret_cast<const unsigned long long*>(gnodes) + i);
        for (int i = l; i < np * 5; i += 32)
            reinterpret_cast<unsigned long long*>(pend)[i] = __ldcg(reinterpret_cast<const unsigned long long*>(gpend) + i);
        for (int i = l; i < eh.avail * M; i += 32) {
            ltok[i] = __ldcg(gl + 2 * i);
            lprob[i] = __int_as_float(__ldcg(gl + 2 * i + 1));
        }
    }
    __syncwarp();
    if (!trivial) {
        const int S = task_S(A, job.task);
        load_hdrs_w(A.W, b, S, sh.hdrs);
        uint32_t flags = l < S ? sh.hdrs.flags[l] : 0u;
        uint64_t theta = l < S ? sh.hdrs.kth[l] : 0ull;
        flags = __reduce_or_sync(0xffffffffu, flags);
        theta = warp_max_u64(theta);
        int n = 0;
        if (flags & kPfBad) {
            n = 0;
        } else if (flags & kPfOverflow) {
            const float* qrow = A.q + static_cast<long long>(b) * A.q_bs + static_cast<long long>(d - 1) * A.q_rs;
            n = build_fallback(qrow, A.V, M, list);
        } else {
            // every slice key at or above the largest slice filter, then the top M
            bool of;
            n = gather_keys_w(A.W, b, S, sh.hdrs, [&](uint64_t key) { return key >= theta; }, list, kBuildList, of);
            if (n > M) {
                const uint64_t kth = kth_key_w(list, n, M);
                // keep the keys >= kth (exactly M: composite keys are unique)
                const uint32_t lt = (1u << l) - 1u;
                int out = 0;
                for (int i0 = 0; i0 < n; i0 += 32) {
                    const int i = i0 + l;
                    uint64_t key = 0;
                    bool p = false;
                    if (i < n) { key = list[i]; p = key >= kth; }
                    const uint32_t bal = __ballot_sync(0xffffffffu, p);
                    if (p) list[out + __popc(bal & lt)] = key;
                    out += __popc(bal);
                }
                __syncwarp();
                n = out;
            }
        }
        // the depth list in rank order (value desc, index asc)
        for (int i = l; i < n; i += 32) {
            const uint64_t key = list[i];
            int r = 0;
            for (int j = 0; j < n; ++j) r += list[j] > key;
            const int o = (d - 1) * M + r;
            ltok[o] = ckey_idx(key);
            lprob[o] = ckey_val(key);
            __stcg(gl + 2 * o, ckey_idx(key));
            __stcg(gl + 2 * o + 1, __float_as_int(ckey_val(key)));
        }
        if (l == 0) {
            eh.len[d] = n;
            eh.avail = d;
            if (flags & kPfBad) eh.status |= 1;
        }
        __syncwarp();
    }
    // ---- best-first enumeration (lane 0), resumable ----
    int need = 0;
    if (l == 0) {
        int count = eh.count, np = eh.npend, want = eh.want;
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
    }
    need = __shfl_sync(0xffffffffu, need, 0);
    __syncwarp();
    if (need == 0) {
        build_finalize(A, msk, nodes, ltok, b, eh.count, eh.status);
    } else {
        // save the state and ask for depth `need`
        const int nc = eh.count, np = eh.npend;
        for (int i = l; i < nc * 5; i += 32)
            __stcg(reinterpret_cast<unsigned long long*>(gnodes) + i, reinterpret_cast<const unsigned long long*>(nodes)[i]);
        for (int i = l; i < np * 5; i += 32)
            __stcg(reinterpret_cast<unsigned long long*>(gpend) + i, reinterpret_cast<const unsigned long long*>(pend)[i]);
        for (int i = l; i < static_cast<int>(sizeof(EnumHdr) / 4); i += 32)
            __stcg(reinterpret_cast<int*>(gh) + i, reinterpret_cast<const int*>(&eh)[i]);
        __syncwarp();
        if (l == 0) {
            Task nt;
            nt.b = b; nt.row = need - 1; nt.kind = 0; nt.aux = 0; nt.st = 0; nt.base = base;
            int S1, SL1;
            pick_slices(A.B, A.V, A.S, A.S1, done, S1, SL1);
            push_task(A.W, nt, S1, SL1, true);   // the next combine reads the saved state
        }
    }
    __syncwarp();
}

__global__ void __launch_bounds__(kBlockThreads, kCtasPerSm) build_kernel(const BuildArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    auto& sh = *reinterpret_cast<BuildSmem*>(smem + kStages * kChunkBytes);
    unsigned char* scr = smem + kStages * kChunkBytes + sizeof(BuildSmem);
    Ent* nodes = reinterpret_cast<Ent*>(scr + build_scr_bytes(A.N, A.L));
    Ent* pend = nodes + A.N;
    if (threadIdx.x == 0) topk_smem_init(sh.tk);   // made visible by pipe_init's barrier
    const Pipe P = pipe_init(smem, sh.pipe);
    const int N = A.N, M = A.M, L = A.L;
    const bool tma = A.tma_q != 0;
    auto trivial_of = [&](const Task& t) { return t.kind < 0 && (N <= 1 || L <= 0); };
    auto plan = [&](const Task& t, int slice) {
        if (trivial_of(t)) return plan_none();
        const int SL = task_SL(A, t);
        const int x0 = slice * SL, x1 = min(A.V, x0 + SL);
        const float* qrow = A.q + static_cast<long long>(t.b) * A.q_bs + static_cast<long long>(t.row) * A.q_rs;
        return plan_single(qrow, 4, x0, x1);
    };
    if (threadIdx.x >= kCombiner0) {
        combiner_loop(P, [&](const Job& job) {
            uint32_t done;
            uint32_t base;
            if (comb_arrive(A.W, job.task, task_S(A, job.task), &done, &base))
                build_combine(A, sh, scr, nodes, pend, job, done, base);
            __syncwarp();
        });
        return;
    }
    if (threadIdx.x >= kThreads) {
        if (threadIdx.x == kProducer)
            producer_loop(A.W, A.B, A.S, P, tma, [](Claimed&) {},
                          [&](const Claimed& c) { return plan(c.task, c.slice); });
        return;
    }
    uint32_t seq = 0, jseq = 0, cseq = 0;
    auto serve = []() {};   // every combine runs on the combiner warp
    for (uint32_t u = 0;; ++u) {
        const Claimed cl = next_unit(P, u, cseq, serve);
        if (!cl.ok) break;
        const Task t = cl.task;
        const int s = cl.slice;
        const int b = t.b;
        const bool trivial = trivial_of(t);
        PartHdr* ph = part_hdr(A.W, b, s, A.S);
        uint64_t* pk = part_keys(A.W, b, s, A.S);
        if (!trivial) {
            const int x0 = s * task_SL(A, t);
            TopkHistFn<F32, false> fn;
            fn.init(&sh.tk, M, 0u, u + 1u);
            if (!consume_row<F32>(P, seq, plan(t, s), tma, x0, fn)) break;
            uint64_t F;
            uint32_t oflow, bad;
            float vm;
            int n = fn.finish(F, oflow, bad, vm);
            uint64_t* list = sh.tk.cand;
            if (n > A.cap_p && !bad && !oflow) {
                // the slice's exact M-th key: a certified value bound, then the
                // index bits within that value
                // (repeated until it stops rising: then it is the exact M-th value)
                for (int it = 0; it < 8 && n > A.cap_p; ++it) {
                    bool cert;
                    const uint32_t F2 = hist_bound_list(list, n, M, hkey(F), sh.hist, sh.scratch, cert);
                    if (!(cert && F2 > hkey(F))) break;
                    n = compact_list(list, n, F2, sh.ired);
                    F = static_cast<uint64_t>(F2) << 32;
                }
                if (n > A.cap_p) {
                    const uint64_t kth = composite_bound(
                        [&](auto f) { for (int i = threadIdx.x; i < n; i += kThreads) f(list[i]); },
                        M, F, sh.ired);
                    // keep the keys >= kth (order kept)
                    int out = 0;
                    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
                    for (int i0 = 0; i0 < n; i0 += kThreads) {
                        const int i = i0 + threadIdx.x;
                        uint64_t key = 0;
                        bool p = false;
                        if (i < n) { key = list[i]; p = key >= kth; }
                        const uint32_t bal = __ballot_sync(0xffffffffu, p);
                        if (lane == 0) sh.ired[w] = __popc(bal);
                        csync();
                        int base = out, tot = 0;
                        for (int j = 0; j < kWarps; ++j) {
                            if (j < w) base += sh.ired[j];
                            tot += sh.ired[j];
                        }
                        csync();
                        if (p) list[base + __popc(bal & ((1u << lane) - 1u))] = key;
                        out += tot;
                        csync();
                    }
                    n = out;
                    F = kth;
                    if (n > A.cap_p) oflow = 1;
                }
            }
            if (bad || oflow) n = 0;
            csync();
            for (int i = threadIdx.x; i < n; i += kThreads) __stcg(pk + i, list[i]);
            if (threadIdx.x == 0) {
                ph->flags = (bad ? kPfBad : 0u) | (oflow ? kPfOverflow : 0u);
                ph->cnt = n;
                ph->kth = F;
            }
        }
        csync();
        Job j;
        j.task = t; j.slice = s; j.kind = trivial ? 1 : 0; j.stop = 0; j.flags = 0;
        post_job(P, jseq, cseq, j, serve);
    }
    Job j;
    j.task.b = 0; j.task.row = 0; j.task.kind = 0; j.task.aux = 0; j.task.st = 0; j.task.base = 0;
    j.slice = 0; j.kind = 0; j.stop = 1; j.flags = 0;
    post_job(P, jseq, cseq, j, serve);
}

// largest slice count whose candidate lists fit the combine's gather buffer
int build_max_slices(int N, int L) {
    (void)L;
    const int M = N - 1;
    // the combiner warp merges every slice's list: keep that under ~8 lists
    int s = M > 0 ? kBuildList / M : kMaxSlices;
    if (s > 8) s = 8;
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
