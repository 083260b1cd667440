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
// best-first enumeration then runs on the leader's combiner warp.  The
// frontier is kept per emitted node: every node carries the head of its
// children not emitted yet (the next rank of the next depth's list, with its
// Q), so the frontier is the set of heads, and each pop -- a warp-wide
// arg-max over the nodes' heads -- emits one head as a new node, advances its
// parent's head to the next rank and gives the new node its first head (rank
// 0 of the next depth).  A node's successors score no higher than it (q <=
// 1), so pops come out in non-increasing Q and the first `budget` pops are
// the best prefixes.  When a first child needs a depth
// whose list is not built yet, the enumeration saves its state to the
// workspace and posts that depth's row job; depth rows past the last one the
// enumeration consults are never read.
#include "spec_chain.cuh"
#include "spec_select.cuh"

namespace spec {

struct Ent {                 // an emitted node and the head of its children
    double Q;
    double hq;               // Q of its next child not emitted yet (< 0: none, or not known yet)
    unsigned long long ph, pl;   // rank path, one byte per depth, depth 1 in the top byte
    int depth, parent, rank;
    int next;                // the rank of that child in the next depth's list
};
static_assert(sizeof(Ent) == 48, "Ent is 48 bytes");

struct EnumHdr {
    int count, unused, want, avail;
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
    uint32_t last_hint;      // combiner: value filter hint for the next row (0: none)
    uint32_t depth_hint[17]; // DDTree: the hint for depth d's rows (index 1..16; 0: none)
    alignas(16) uint64_t list[kBuildList];   // combiner: gathered keys
};

// Filter hints for top-M rows of probabilities: half of the last row's M-th
// largest value (rows of one drafter differ little in it; a hint above a
// row's M-th value costs a second pass over that row).  Kept across calls in
// the workspace, tagged with V and M.
constexpr uint32_t kPersistTagTopm = 0x5e1ec7eeu;
__device__ __forceinline__ uint32_t topm_hint(float vM) { return vM > 0.f ? fkey(0.5f * vM) : 0u; }
__device__ __forceinline__ uint32_t topm_hint_load(const Ctrl* ctrl, int V, int M) {
    const uint4 ps = __ldcg(reinterpret_cast<const uint4*>(ctrl->persist + 4));
    return (ps.x == kPersistTagTopm && ps.z == static_cast<uint32_t>(V) && ps.w == static_cast<uint32_t>(M)) ? ps.y
                                                                                                           : 0u;
}
__device__ __forceinline__ void topm_hint_store(Ctrl* ctrl, uint32_t h, int V, int M) {
    __stcg(reinterpret_cast<uint4*>(ctrl->persist + 4),
           make_uint4(kPersistTagTopm, h, static_cast<uint32_t>(V), static_cast<uint32_t>(M)));
}
// DDTree rows differ by depth (a drafter's position-d distributions are alike
// across requests, not across depths): one hint per depth, from the last
// depth-d row a CTA merged, and kept across calls (persist[8..10] tag, V, M;
// persist[11 + d - 1] depth d's hint).
constexpr uint32_t kPersistTagDepth = 0x5e1ec7efu;
__device__ __forceinline__ void depth_hints_load(const Ctrl* ctrl, int V, int M, int L, uint32_t* dh) {
    const bool ok = __ldcg(ctrl->persist + 8) == kPersistTagDepth &&
                    __ldcg(ctrl->persist + 9) == static_cast<uint32_t>(V) &&
                    __ldcg(ctrl->persist + 10) == static_cast<uint32_t>(M);
    dh[0] = 0u;
    for (int d = 1; d <= 16; ++d) dh[d] = (ok && d <= L) ? __ldcg(ctrl->persist + 10 + d) : 0u;
}
__device__ __forceinline__ void depth_hint_store(Ctrl* ctrl, int d, uint32_t h, int V, int M) {
    __stcg(ctrl->persist + 8, kPersistTagDepth);
    __stcg(ctrl->persist + 9, static_cast<uint32_t>(V));
    __stcg(ctrl->persist + 10, static_cast<uint32_t>(M));
    __stcg(ctrl->persist + 10 + d, h);
}

// per-request workspace: [EnumHdr][lists L*M (tok, prob bits)][nodes N]
__host__ __device__ inline size_t build_lists_off() { return 128; }
__host__ __device__ inline size_t build_nodes_off(int N, int L) {
    return (build_lists_off() + static_cast<size_t>(L) * (N - 1) * 8 + 127) & ~static_cast<size_t>(127);
}
size_t build_extra_bytes(int N, int L) {
    return (build_nodes_off(N, L) + static_cast<size_t>(N) * sizeof(Ent) + 127) & ~static_cast<size_t>(127);
}
// combiner shared memory after the partial areas: depth lists and nodes
__host__ __device__ inline size_t enum_smem_bytes(int N, int L) {
    return ((static_cast<size_t>(L) * (N - 1) * 8 + 15) & ~static_cast<size_t>(15)) +
           static_cast<size_t>(N) * sizeof(Ent);
}

// rank path with byte d set to r (depth 1 in the top byte of ph)
__device__ __forceinline__ void path_with(unsigned long long& ph, unsigned long long& pl, int d, int r) {
    const unsigned long long v = static_cast<unsigned long long>(r & 0xff);
    if (d <= 8) {
        const int sh = 8 * (8 - d);
        ph = (ph & ~(0xffull << sh)) | (v << sh);
    } else {
        const int sh = 8 * (16 - d);
        pl = (pl & ~(0xffull << sh)) | (v << sh);
    }
}

// the enumeration's shared-memory view (combiner warp): depth lists
// (tokens, probabilities), emitted nodes, frontier
struct EnumView {
    int* ltok;
    float* lprob;
    Ent* nodes;
    uint32_t a_lprob, a_nodes;   // the same, as shared-window addresses
};

// Ent records through shared-window addresses (explicit shared loads and
// stores: the enumeration's records are reached through struct members,
// which would otherwise be generic accesses)
__device__ __forceinline__ uint64_t ldsv_u64(uint32_t a) {
    uint64_t v;
    asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void stsv_u64(uint32_t a, uint64_t v) {
    asm volatile("st.shared.u64 [%0], %1;" :: "r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ EnumView enum_view(unsigned char* base, int N, int L) {
    EnumView v;
    const int LM = L * (N - 1);
    v.ltok = reinterpret_cast<int*>(base);
    v.lprob = reinterpret_cast<float*>(base + static_cast<size_t>(LM) * 4);
    v.nodes = reinterpret_cast<Ent*>(base + ((static_cast<size_t>(LM) * 8 + 15) & ~static_cast<size_t>(15)));
    v.a_lprob = smem_u32(v.lprob);
    v.a_nodes = smem_u32(v.nodes);
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

// The frontier's best head, on the combiner warp.  Node n belongs to lane
// n % 32; each lane keeps the best head among its nodes in registers and
// recomputes it only when one of its nodes changed.  Heads are ordered by Q
// (descending), then by the child's depth (ascending), then by the child's
// rank path (ascending); Q is compared through an order-preserving 64-bit key
// of the double, and the rest only among exact ties.
__device__ __forceinline__ unsigned long long q_order_key(unsigned long long qb) {
    if ((qb << 1) == 0ull) qb = 0ull;                              // -0 as +0
    return (qb >> 63) ? ~qb : (qb | 0x8000000000000000ull);
}
// a node without a head stores hq = -1.0
constexpr unsigned long long kNoHead = 0xbff0000000000000ull;
// head key of a node from its hq bits: 0 when it has no head (integer tests:
// the fp64 pipe is narrow on this part)
__device__ __forceinline__ unsigned long long head_key_bits(unsigned long long hb) {
    return hb == kNoHead ? 0ull : q_order_key(hb);
}
__device__ __forceinline__ unsigned long long head_key(uint32_t a_node) {
    return head_key_bits(ldsv_u64(a_node + offsetof(Ent, hq)));
}
// the child path and depth a head stands for
__device__ __forceinline__ void head_path(uint32_t a_node, int& d, unsigned long long& ph, unsigned long long& pl) {
    const uint64_t dp = ldsv_u64(a_node + offsetof(Ent, depth));     // depth, parent
    const uint64_t rn = ldsv_u64(a_node + offsetof(Ent, rank));      // rank, next
    ph = ldsv_u64(a_node + offsetof(Ent, ph));
    pl = ldsv_u64(a_node + offsetof(Ent, pl));
    d = static_cast<int>(static_cast<uint32_t>(dp)) + 1;
    path_with(ph, pl, d, static_cast<int>(static_cast<uint32_t>(rn >> 32)));
}
// exact-tie order of two heads with equal Q keys: depth, then rank path
__device__ __noinline__ bool head_before_tie(uint32_t a1, uint32_t a2) {
    int d1, d2;
    unsigned long long h1, l1, h2, l2;
    head_path(a1, d1, h1, l1);
    head_path(a2, d2, h2, l2);
    if (d1 != d2) return d1 < d2;
    if (h1 != h2) return h1 < h2;
    return l1 < l2;
}
struct LaneBest {
    int j;                   // node, -1: none
    unsigned long long k;    // its head key
};
__device__ __forceinline__ void lane_best(uint32_t a_nodes, int count, LaneBest& b) {
    const int l = threadIdx.x & 31;
    constexpr uint32_t kE = static_cast<uint32_t>(sizeof(Ent));
    b.j = -1; b.k = 0;
    for (int j = l; j < count; j += 32) {
        const unsigned long long k = head_key(a_nodes + kE * j);
        if (k == 0ull) continue;
        if (b.j < 0 || k > b.k || (k == b.k && head_before_tie(a_nodes + kE * j, a_nodes + kE * b.j))) {
            b.j = j;
            b.k = k;
        }
    }
}
__device__ __forceinline__ int warp_best(const LaneBest& b, uint32_t a_nodes) {
    const int l = threadIdx.x & 31;
    uint32_t cand;
    {
        // every head key has its top bit set: 0 stands for no head
        const uint32_t hi = b.j >= 0 ? static_cast<uint32_t>(b.k >> 32) : 0u;
        const uint32_t m = __reduce_max_sync(0xffffffffu, hi);
        if (m == 0u) return -1;
        cand = __ballot_sync(0xffffffffu, hi == m);
    }
    if (__popc(cand) > 1) {
        const bool in = (cand >> l) & 1u;
        const uint32_t lo = static_cast<uint32_t>(b.k);
        const uint32_t m = __reduce_max_sync(0xffffffffu, in ? lo : 0u);
        cand = __ballot_sync(0xffffffffu, in && lo == m);
    }
    int best = __shfl_sync(0xffffffffu, b.j, __ffs(cand) - 1);
    if (__popc(cand) > 1) {
        // exact ties in Q: the order on depth and rank path, over the tied lanes
        constexpr uint32_t kE = static_cast<uint32_t>(sizeof(Ent));
        cand &= cand - 1u;
        while (cand) {
            const int j = __shfl_sync(0xffffffffu, b.j, __ffs(cand) - 1);
            if (head_before_tie(a_nodes + kE * j, a_nodes + kE * best)) best = j;
            cand &= cand - 1u;
        }
    }
    return best;
}

// The best-first enumeration from the saved state in `eh` / `ev` (combiner
// warp).  Returns the depth whose list it needs next, or 0 when the tree is
// complete.
__device__ int enumerate_w(const BuildArgs& A, EnumHdr& eh, const EnumView& ev) {
    const int l = threadIdx.x & 31;
    const int N = A.N, M = A.M, L = A.L;
    int count = eh.count, want = eh.want;
    const int avail = eh.avail;
    const int lenl = l <= L ? eh.len[l] : 0;          // lane d: depth d's list length
    int need = 0;
    constexpr uint32_t kE = static_cast<uint32_t>(sizeof(Ent));
    // scalar copies: the explicit shared accesses below clobber memory, and a
    // view reached through a reference would be reloaded after every one
    const uint32_t a_lprob = ev.a_lprob, a_nodes = ev.a_nodes;
    auto lprob_at = [a_lprob](int i) { return __uint_as_float(lds_u32(a_lprob + 4u * static_cast<uint32_t>(i))); };
    auto st_f64 = [](uint32_t a, double v) { stsv_u64(a, static_cast<uint64_t>(__double_as_longlong(v))); };
    auto ld_f64 = [](uint32_t a) { return __longlong_as_double(static_cast<long long>(ldsv_u64(a))); };
#ifdef SPEC_TRACE
    long long t_best = 0, t_upd = 0, t_lb = 0;
    const long long t_all = clock64();
#endif
    // a node of an earlier call whose first head waited for its depth's list
    if (want >= 0 && count < N) {
        const uint32_t aw = a_nodes + kE * want;
        const int dd = static_cast<int>(static_cast<uint32_t>(ldsv_u64(aw + offsetof(Ent, depth)))) + 1;
        if (dd <= L) {
            if (dd > avail) {
                need = dd;
            } else {
                const bool has = __shfl_sync(0xffffffffu, lenl, dd) > 0;
                const double hq = has ? ld_f64(aw + offsetof(Ent, Q)) * static_cast<double>(lprob_at((dd - 1) * M))
                                      : -1.0;
                if (l == (want & 31)) st_f64(aw + offsetof(Ent, hq), hq);
            }
        }
        if (!need) want = -1;
    }
    __syncwarp();
    LaneBest lb;
    lane_best(a_nodes, count, lb);
    while (!need && count < N) {
#ifdef SPEC_TRACE
        const long long tq0 = clock64();
#endif
        const int v = warp_best(lb, a_nodes);
#ifdef SPEC_TRACE
        t_best += clock64() - tq0;
#endif
        if (v < 0) break;
        // the head of v becomes node c: its Q, depth, rank and path; v's
        // head moves to its next rank, c's first head is rank 0 of the next
        // depth (independent loads, independent products)
        const uint32_t av = a_nodes + kE * v;
        const double Qv = ld_f64(av + offsetof(Ent, Q));
        const double Qc = ld_f64(av + offsetof(Ent, hq));
        const uint64_t dp = ldsv_u64(av + offsetof(Ent, depth));
        const uint64_t rn = ldsv_u64(av + offsetof(Ent, rank));
        unsigned long long ph = ldsv_u64(av + offsetof(Ent, ph)), pl = ldsv_u64(av + offsetof(Ent, pl));
        const int d = static_cast<int>(static_cast<uint32_t>(dp)) + 1;
        const int r = static_cast<int>(static_cast<uint32_t>(rn >> 32));
        const bool deeper = d + 1 <= L;
        // the list lengths and both probabilities at once (clamped indices:
        // the loads do not wait for the tests)
        const int len_d = __shfl_sync(0xffffffffu, lenl, d);
        const int len_n = __shfl_sync(0xffffffffu, lenl, deeper ? d + 1 : 0);
        const float qs = lprob_at((d - 1) * M + min(r + 1, M - 1));
        const float q0 = lprob_at(deeper ? d * M : 0);
        const bool sib = r + 1 < len_d;
        const bool have_list = deeper && d + 1 <= avail && len_n > 0;
        const double hv = sib ? Qv * static_cast<double>(qs) : -1.0;
        const double hc = have_list ? Qc * static_cast<double>(q0) : -1.0;
        path_with(ph, pl, d, r);
        const int nid = count++;
        const uint32_t ac = a_nodes + kE * nid;
        // every lane stores the same values (no divergent branch; a warp's
        // stores of one value to one address are one write)
        st_f64(av + offsetof(Ent, hq), hv);
        stsv_u64(av + offsetof(Ent, rank), (static_cast<uint64_t>(r + 1) << 32) | static_cast<uint32_t>(rn));
        st_f64(ac + offsetof(Ent, Q), Qc);
        st_f64(ac + offsetof(Ent, hq), hc);
        stsv_u64(ac + offsetof(Ent, ph), ph);
        stsv_u64(ac + offsetof(Ent, pl), pl);
        stsv_u64(ac + offsetof(Ent, depth), (static_cast<uint64_t>(static_cast<uint32_t>(v)) << 32) |
                                                static_cast<uint32_t>(d));
        stsv_u64(ac + offsetof(Ent, rank), static_cast<uint32_t>(r));   // next = 0
        if (deeper && count < N && d + 1 > avail) {
            // c's first head needs a depth not read yet: stop, and resume here
            want = nid;
            need = d + 1;
        }
#ifdef SPEC_TRACE
        __syncwarp();
        const long long tq1 = clock64();
        t_upd += tq1 - tq0;
#endif
        // every lane recomputes its best over its nodes (only the two lanes
        // owning v and the new node find a change; running it everywhere
        // keeps the warp converged)
        __syncwarp();
        lane_best(a_nodes, count, lb);
#ifdef SPEC_TRACE
        t_lb += clock64() - tq1;
#endif
    }
#ifdef SPEC_TRACE
    if (l == 0) SPEC_TRACE_EV(16, static_cast<int>(t_best), static_cast<int>(clock64() - t_all), count);
    if (l == 0) SPEC_TRACE_EV(17, static_cast<int>(t_upd), static_cast<int>(t_lb), 0);
#endif
    __syncwarp();
    if (l == 0) { eh.count = count; eh.want = want; }
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
    const int nc = eh.count;
    constexpr int kW = static_cast<int>(sizeof(Ent) / 8);
    for (int i = l; i < nc * kW; i += 32)
        __stcg(reinterpret_cast<unsigned long long*>(ex + build_nodes_off(N, L)) + i,
               reinterpret_cast<const unsigned long long*>(ev.nodes)[i]);
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
    const int nc = eh.count;
    constexpr int kW = static_cast<int>(sizeof(Ent) / 8);
    for (int i = l; i < nc * kW; i += 32)
        reinterpret_cast<unsigned long long*>(ev.nodes)[i] =
            __ldcg(reinterpret_cast<const unsigned long long*>(ex + build_nodes_off(N, L)) + i);
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
__device__ int merge_sorted_topm_w(const unsigned char* parts, int pb, int C, int M, int cnt, int* tok, float* prob);

struct BuildOp {
    using Args = BuildArgs;
    using Smem = BuildSmem;

    __device__ static int batch(const Args& A) { return A.B; }
    __device__ static bool tma(const Args& A) { return A.tma_q != 0; }
    __device__ static void prefetch(const Args&, const Geo&, Job&, Smem&) {}
    __device__ static void init_smem(const Args& A, const Geo&, Smem& sm) {
        if (threadIdx.x == 0) {
            topk_smem_init(sm.tk);
            sm.last_hint = 0u;
            depth_hints_load(A.E.W.ctrl, A.V, A.M, A.L, sm.depth_hint);
        }
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
            h.count = 1; h.want = 0; h.avail = 0; h.status = 0;
            eh = h;
            Ent root{};
            root.Q = 1.0; root.hq = -1.0; root.depth = 0; root.parent = -1; root.rank = -1; root.next = 0;
            ev.nodes[0] = root;
        }
        __syncwarp();
        if (A.N <= 1 || A.L <= 0) {
            build_finalize(A, ev, b, 1, 0);
            return job_done();
        }
        if (G.own > 1) enum_save(A, b, eh, ev, 0);
        Job j = make_job(b, 0, 0, 0);   // depth 1's row
        j.hint = sm.depth_hint[1];
        return j;
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
        fn.init(&sm.tk, M, j.hint, seq + 1u);   // every consumer holds the same seq
        if (!consume_row<F32>(P, seq, plan(A, G, j), tma, slice_x0(G, G.rank), fn)) return -1;
        SPEC_TRACE_T(tf0);
        uint64_t F;
        uint32_t oflow, bad;
        float vm;
        int n = fn.finish(F, oflow, bad, vm);
        SPEC_TRACE_T(tf1);
#ifdef SPEC_TRACE
        const int n_fin = n;
#endif
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
        SPEC_TRACE_T(tf2);
        csync();
        // the keys sorted descending (composite keys are unique: a key's
        // position is the number of greater keys), so that the combine merges
        // sorted lists
        for (int i = threadIdx.x; i < n; i += kThreads) {
            const uint64_t x = list[i];
            int r = 0;
#pragma unroll 8
            for (int j = 0; j < n; ++j) r += list[j] > x ? 1 : 0;
            pk[r] = x;
        }
        if (threadIdx.x == 0) {
            ph->flags = (bad ? kPfBad : 0u) | (oflow ? kPfOverflow : 0u) | (j.hint ? kPfHinted : 0u);
            ph->cnt = n;
            ph->kth = F;
            SPEC_TRACE_EV(24, static_cast<int>(tf1 - tf0), static_cast<int>(tf2 - tf1), static_cast<int>(clock64() - tf2));
            SPEC_TRACE_EV(25, n_fin, n, 0);
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
        SPEC_TRACE_T(tb0);
        const int l = threadIdx.x & 31;
        const int M = A.M, C = G.C, pb = G.part_bytes;
        const int b = j.b;
        const int d = j.row + 1;
        const EnumView ev = view(A, G);
        EnumHdr& eh = sm.eh;
        // a CTA that leads one slot keeps its request's enumeration in shared
        // memory between jobs; with several slots it is saved in the workspace
        if (G.own > 1) enum_load(A, b, eh, ev);
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
        int n;
        if (!(flags & (kPfBad | kPfOverflow))) {
            // the depth list in rank order (value desc, index asc) from the
            // slices' sorted lists
            n = merge_sorted_topm_w(parts, pb, C, M, cnt, ev.ltok + (d - 1) * M, ev.lprob + (d - 1) * M);
        } else {
            n = merge_topm_w(parts, pb, C, M, flags, theta, cnt, qrow, A.V, list);
            for (int i = l; i < n; i += 32) {
                const uint64_t key = list[i];
                int r = 0;
                for (int q = 0; q < n; ++q) r += list[q] > key;
                const int o = (d - 1) * M + r;
                ev.ltok[o] = ckey_idx(key);
                ev.lprob[o] = ckey_val(key);
            }
        }
        if ((flags & kPfHinted) && !(flags & kPfBad) && n < min(M, A.V)) {
            // a hint above this row's M-th value: the row again, unhinted
            return make_job(b, d - 1, 0, 0);
        }
        if (n > 0 && !(flags & kPfBad)) {
            const uint32_t h = topm_hint(ev.lprob[(d - 1) * M + n - 1]);
            if (l == 0) {
                sm.depth_hint[d] = h;
                depth_hint_store(A.E.W.ctrl, d, h, A.V, M);
            }
        }
        if (l == 0) {
            eh.len[d] = n;
            eh.avail = d;
            if (flags & kPfBad) eh.status |= 1;
        }
        __syncwarp();
        SPEC_TRACE_T(tb1);
#ifdef SPEC_TRACE
        const int count0 = eh.count;
#endif
        const int need = enumerate_w(A, eh, ev);
#ifdef SPEC_TRACE
        if (l == 0) SPEC_TRACE_EV(15, static_cast<int>(tb1 - tb0), static_cast<int>(clock64() - tb1), eh.count - count0);
#endif
        if (need == 0) {
            build_finalize(A, ev, b, eh.count, eh.status);
            return job_done();
        }
        if (G.own > 1) enum_save(A, b, eh, ev, d - 1);
        Job nj = make_job(b, need - 1, 0, 0);
        nj.hint = sm.depth_hint[need];
        return nj;
    }
};

// The row's top-M from the slices' sorted lists (combiner warp), written to
// tok / prob in rank order: a key's merged rank is the number of greater keys
// over all lists (binary searches, kRegKeys keys per lane at a time, every
// load unconditional so that a step's loads issue together); the keys of
// rank < M are the row's M largest.  `cnt`: lane r holds list r's length.
// Returns min(total, M).
constexpr int kMergeKeys = 4;
__device__ int merge_sorted_topm_w(const unsigned char* parts, int pb, int C, int M, int cnt, int* tok,
                                   float* prob) {
    const int l = threadIdx.x & 31;
    const int cl = l < C ? cnt : 0;
    int tot;
    const int off = warp_exscan_i(cl, tot);
    if (tot == 0) return 0;
    const uint32_t kb0 = smem_u32(parts) + static_cast<uint32_t>(sizeof(PartHdr));
    const uint32_t mmax = warp_max_u32(static_cast<uint32_t>(cl));
    const int s0 = 1 << (31 - __clz(mmax));
    if (C <= 4) {
        // every search of every key at once (lists q >= C are empty): one
        // step's loads for all lists and keys issue together, so a pass costs
        // log2(list length) dependent steps instead of C times as many
        int o[4], mq[4];
        uint32_t lb[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            o[q] = q < C ? __shfl_sync(0xffffffffu, off, q) : tot;
            mq[q] = __shfl_sync(0xffffffffu, cl, q);
            lb[q] = kb0 + static_cast<uint32_t>((q < C ? q : 0) * pb);
        }
        for (int f0 = 0; f0 < tot; f0 += 32 * kMergeKeys) {
            uint64_t key[kMergeKeys];
#pragma unroll
            for (int j = 0; j < kMergeKeys; ++j) {
                const int f = min(f0 + l + 32 * j, tot - 1);
                const int r = (f >= o[1] ? 1 : 0) + (f >= o[2] ? 1 : 0) + (f >= o[3] ? 1 : 0);
                const int base = r == 0 ? 0 : (r == 1 ? o[1] : (r == 2 ? o[2] : o[3]));
                key[j] = lds_u64(kb0 + static_cast<uint32_t>(r * pb + (f - base) * 8));
            }
            int pos[4][kMergeKeys];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < kMergeKeys; ++j) pos[q][j] = 0;
            for (int st = s0; st > 0; st >>= 1) {
                uint64_t v[4][kMergeKeys];
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int j = 0; j < kMergeKeys; ++j)
                        v[q][j] = lds_u64(lb[q] + static_cast<uint32_t>((max(min(pos[q][j] + st, mq[q]), 1) - 1) * 8));
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int j = 0; j < kMergeKeys; ++j) {
                        const int np = pos[q][j] + st;
                        pos[q][j] = (np <= mq[q] && v[q][j] > key[j]) ? np : pos[q][j];
                    }
            }
#pragma unroll
            for (int j = 0; j < kMergeKeys; ++j) {
                const int rank = pos[0][j] + pos[1][j] + pos[2][j] + pos[3][j];
                if (f0 + l + 32 * j < tot && rank < M) {
                    tok[rank] = ckey_idx(key[j]);
                    prob[rank] = ckey_val(key[j]);
                }
            }
        }
        __syncwarp();
        return tot < M ? tot : M;
    }
    for (int f0 = 0; f0 < tot; f0 += 32 * kMergeKeys) {
        uint64_t key[kMergeKeys];
        int rank[kMergeKeys];
#pragma unroll
        for (int j = 0; j < kMergeKeys; ++j) {
            const int f = min(f0 + l + 32 * j, tot - 1);
            int r = 0;
            for (int q = 1; q < C; ++q) r += __shfl_sync(0xffffffffu, off, q) <= f ? 1 : 0;
            const int base = __shfl_sync(0xffffffffu, off, r);
            key[j] = lds_u64(kb0 + static_cast<uint32_t>(r * pb + (f - base) * 8));
            rank[j] = 0;
        }
        for (int q = 0; q < C; ++q) {
            const int mq = __shfl_sync(0xffffffffu, cl, q);
            const uint32_t lb = kb0 + static_cast<uint32_t>(q * pb);
            int pos[kMergeKeys];
#pragma unroll
            for (int j = 0; j < kMergeKeys; ++j) pos[j] = 0;
            for (int st = s0; st > 0; st >>= 1) {
                uint64_t v[kMergeKeys];
#pragma unroll
                for (int j = 0; j < kMergeKeys; ++j)
                    v[j] = lds_u64(lb + static_cast<uint32_t>((max(min(pos[j] + st, mq), 1) - 1) * 8));
#pragma unroll
                for (int j = 0; j < kMergeKeys; ++j) {
                    const int np = pos[j] + st;
                    pos[j] = (np <= mq && v[j] > key[j]) ? np : pos[j];
                }
            }
#pragma unroll
            for (int j = 0; j < kMergeKeys; ++j) rank[j] += pos[j];
        }
#pragma unroll
        for (int j = 0; j < kMergeKeys; ++j) {
            if (f0 + l + 32 * j < tot && rank[j] < M) {
                tok[rank[j]] = ckey_idx(key[j]);
                prob[rank[j]] = ckey_val(key[j]);
            }
        }
    }
    __syncwarp();
    return tot < M ? tot : M;
}

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
    __device__ static void init_smem(const Args& A, const Geo&, Smem& sm) {
        if (threadIdx.x == 0) {
            topk_smem_init(sm.tk);
            sm.last_hint = topm_hint_load(A.base.E.W.ctrl, A.base.V, A.base.M);
        }
    }
    __device__ static EagleRowHdr* row_hdr(const Args& A, int u) {
        return reinterpret_cast<EagleRowHdr*>(A.base.E.W.extra + static_cast<size_t>(u) * A.base.E.W.extra_stride);
    }
    __device__ static Job first(const Args& A, const Geo&, int u, Smem& sm) {
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
        Job j = make_job(b, f, 0, 0);
        j.hint = sm.last_hint;
        j.aux2 = A.front_in[static_cast<long long>(b) * A.F + f];   // the frontier node (checked above)
        return j;
    }
    __device__ static StreamPlan plan(const Args& A, const Geo& G, const Job& j) { return BuildOp::plan(A.base, G, j); }
    __device__ static void prefetch(const Args&, const Geo&, Job&, Smem&) {}
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
        const int u = j.b * A.F + j.row;
        EagleRowHdr* h = row_hdr(A, u);
        // the frontier node's score and depth travel with the row's list, so
        // that the grow step reads one header per slot (issued here, used at
        // the end)
        const long long nb = static_cast<long long>(j.b) * A.G + j.aux2;
        const double psc = A.score[nb];
        const int pdp = A.depth[nb];
        int* tok = reinterpret_cast<int*>(h + 1);
        float* prob = reinterpret_cast<float*>(tok + M);
        int n;
        if (!(flags & (kPfBad | kPfOverflow))) {
            n = merge_sorted_topm_w(parts, pb, C, M, cnt, tok, prob);
            if ((flags & kPfHinted) && n < min(M, A.base.V)) {
                // a hint above this row's K2-th value: the row again, unhinted
                Job r = make_job(j.b, j.row, 0, 0);
                r.aux2 = j.aux2;
                return r;
            }
            if (n > 0) {
                const uint32_t hn = topm_hint(prob[n - 1]);
                if (l == 0) {
                    sm.last_hint = hn;
                    topm_hint_store(A.base.E.W.ctrl, hn, A.base.V, M);
                }
            }
        } else {
            n = merge_topm_w(parts, pb, C, M, flags, theta, cnt, qrow, A.base.V, sm.list);
            for (int i = l; i < n; i += 32) {
                const uint64_t key = sm.list[i];
                int r = 0;
                for (int q = 0; q < n; ++q) r += sm.list[q] > key;
                tok[r] = ckey_idx(key);
                prob[r] = ckey_val(key);
            }
        }
        if (l == 0) {
            h->n = n;
            h->bad = (flags & kPfBad) ? 1 : 0;
            h->node = j.aux2;
            h->depth = pdp;
            h->score = psc;
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

#ifdef SPEC_TRACE
// development builds: this translation unit's event trace buffer
extern "C" int spec_trace_setup_build(void* buf, unsigned cap) {
    unsigned z = 0;
    if (cudaMemcpyToSymbol(spec::g_trace, &buf, sizeof(buf)) != cudaSuccess) return 1;
    if (cudaMemcpyToSymbol(spec::g_trace_cap, &cap, sizeof(cap)) != cudaSuccess) return 1;
    return cudaMemcpyToSymbol(spec::g_trace_n, &z, sizeof(z)) != cudaSuccess;
}
extern "C" unsigned spec_trace_count_build(void) {
    unsigned n = 0;
    cudaMemcpyFromSymbol(&n, spec::g_trace_n, sizeof(n));
    return n;
}
#endif
