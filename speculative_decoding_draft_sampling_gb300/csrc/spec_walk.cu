// spec_walk.cu -- argmax walks on the cluster engine.
//
// [SD-survey] = "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
// (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash, DDTree and
// DSpark), chzhyang.github.io.
//
// Greedy verification (§1, greedy-consistent results): row i's argmax (raw
// logits, lowest id on ties) is compared with draft y_i; a match reads row
// i+1, a mismatch commits the argmax; row k's argmax is the bonus token.
//
// Tree walk (§5 "DDTree"): from the root, the argmax of the current node's
// row is looked up among the node's children; a matching child is accepted
// and becomes the current node; otherwise the argmax is the bonus token.
// Only rows on the walked path are read.
//
// One job per row: every CTA of the cluster reduces its vocabulary slice to
// (max value, lowest index) as a composite key; the slot's leader takes the
// maximum over the slices and decides.
#include "spec_chain.cuh"
#include "spec_select.cuh"

namespace spec {

// combiner: the children of the node a tree walk reads next (ascending id),
// found while its row streams
constexpr int kChildCache = 64;
struct WalkSmem {
    uint64_t red[kWarps];
    uint32_t wb[kWarps];
    int cb, cnode, cn;                 // request, node, children cached (-1: too many)
    int cid[kChildCache];
    int ctok[kChildCache];
};
// a greedy walk job whose combine inputs the combiner loaded ahead
constexpr int kWalkPrefetched = 0x7e1ec8;

template <class E, bool kTree>
__device__ __forceinline__ const void* walk_row(const WalkArgs& A, int b, int i) {
    long long r;
    if (!kTree && A.k_per_req && A.l_row_off) r = static_cast<long long>(A.l_row_off[b] + i) * A.l_rs;
    else r = static_cast<long long>(b) * A.l_bs + static_cast<long long>(i) * A.l_rs;
    return static_cast<const unsigned char*>(A.logits) + r * E::kBytes;
}

// combiner warp: the greedy request's outputs
__device__ Job greedy_finish(const WalkArgs& A, int b, int n, int last, int st) {
    const int W = A.K + 1;
    const int l = threadIdx.x & 31;
    int* out = A.out_tokens + static_cast<long long>(b) * W;
    for (int i = l; i < W; i += 32) {
        int v = -1;
        if (i < n) v = A.draft[static_cast<long long>(b) * A.K + i];
        else if (i == n) v = last;
        out[i] = v;
    }
    if (l == 0) {
        A.num_accepted[b] = n;
        A.status[b] = st;
    }
    __syncwarp();
    return job_done();
}

// combiner warp: the tree walk's outputs; path_nodes[b][1..acc] and
// out_tokens[b][0..acc-1] were written on the way
__device__ Job tree_finish(const WalkArgs& A, int b, int acc, int last, int st) {
    const int W = A.L + 1;
    const int l = threadIdx.x & 31;
    int* pn = A.path_nodes + static_cast<long long>(b) * W;
    int* ot = A.out_tokens + static_cast<long long>(b) * W;
    for (int i = l; i < W; i += 32) {
        if (i > acc) { pn[i] = -1; ot[i] = -1; }
        if (i == acc) ot[i] = last;
    }
    if (l == 0) {
        pn[0] = 0;
        A.num_accepted[b] = acc;
        A.status[b] = st;
    }
    __syncwarp();
    return job_done();
}

template <class E, bool kTree>
struct WalkOp {
    using Args = WalkArgs;
    using Smem = WalkSmem;

    // What the combine reads, loaded by the combiner while the row streams:
    // a greedy walk's draft length and drafted token (into its copy of the
    // job); a tree walk's children of the node (into shared memory).
    __device__ static void prefetch(const Args& A, const Geo&, Job& j, Smem& sm) {
        if (j.b < 0) return;
        const int l = threadIdx.x & 31;
        const int b = j.b, row = j.row;
        if (!kTree) {
            if (l == 0) {
                const int kb = A.k_per_req ? A.k_per_req[b] : A.K;
                j.pad[0] = kb;
                j.y = row < kb && row < A.K ? A.draft[static_cast<long long>(b) * A.K + row] : kYUnknown;
                j.aux2 = kWalkPrefetched;
            }
            __syncwarp();
            return;
        }
        int nn = A.num_nodes[b];
        nn = nn < A.N ? nn : A.N;
        const int* par = A.parent + static_cast<long long>(b) * A.N;
        const int* tok = A.token + static_cast<long long>(b) * A.N;
        const uint32_t lt = (1u << l) - 1u;
        int n = 0;
        for (int c0 = 0; c0 < nn; c0 += 32) {
            const int c = c0 + l;
            const bool is = c < nn && par[c] == row;
            const int t = is ? tok[c] : 0;
            const uint32_t bal = __ballot_sync(0xffffffffu, is);
            const int pos = n + __popc(bal & lt);
            if (is && pos < kChildCache) { sm.cid[pos] = c; sm.ctok[pos] = t; }
            n += __popc(bal);
        }
        if (l == 0) { sm.cb = b; sm.cnode = row; sm.cn = n <= kChildCache ? n : -1; }
        __syncwarp();
    }
    __device__ static int batch(const Args& A) { return A.B; }
    __device__ static bool tma(const Args& A) { return A.tma_l != 0; }
    __device__ static void init_smem(const Args&, const Geo&, Smem& sm) {
        if (threadIdx.x == 0) { sm.cb = -1; sm.cnode = -1; sm.cn = -1; }
    }
    __device__ static Job first(const Args& A, const Geo&, int b, Smem&) {
        if (!kTree) {
            const int kb = A.k_per_req ? A.k_per_req[b] : A.K;
            if (kb < 0 || kb > A.K) return greedy_finish(A, b, 0, -1, 16);
        }
        Job j = make_job(b, 0, 0, 0);
        j.depth = 0;
        return j;
    }
    __device__ static StreamPlan plan(const Args& A, const Geo& G, const Job& j) {
        return plan_single(walk_row<E, kTree>(A, j.b, j.row), E::kBytes, slice_x0(G, G.rank),
                           slice_x1(G, G.rank, A.V), G.chunk);
    }
    __device__ static int consume(const Args& A, const Geo& G, const Pipe& P, uint32_t& seq, bool tma, const Job& j,
                                  Smem& sm, unsigned char* out) {
        PartHdr* ph = reinterpret_cast<PartHdr*>(out);
        ArgmaxFn<E> fn;
        if (!consume_row<E>(P, seq, plan(A, G, j), tma, slice_x0(G, G.rank), fn)) return -1;
        // per warp, then thread 0 over the warps (one barrier)
        const uint64_t wbest = warp_max_u64(fn.key());
        const uint32_t wbad = __reduce_or_sync(0xffffffffu, fn.bad_flag());
        if ((threadIdx.x & 31) == 0) { sm.red[threadIdx.x >> 5] = wbest; sm.wb[threadIdx.x >> 5] = wbad; }
        csync();
        if (threadIdx.x == 0) {
            uint64_t best = 0;
            uint32_t bad = 0;
            for (int q = 0; q < kWarps; ++q) { best = sm.red[q] > best ? sm.red[q] : best; bad |= sm.wb[q]; }
            ph->flags = bad ? kPfBad : 0u;
            ph->kth = best;
            ph->cnt = 0;
        }
        return static_cast<int>(sizeof(PartHdr));
    }
    __device__ static Job combine(const Args& A, const Geo& G, const Job& j, const unsigned char* parts, Smem& sm) {
        const int l = threadIdx.x & 31;
        const int b = j.b, row = j.row;
        int st = j.st;
        uint32_t flags = 0;
        uint64_t best = 0;
        if (l < G.C) {
            const PartHdr* h = part_at(parts, G.part_bytes, l);
            flags = h->flags;
            best = h->kth;
        }
        flags = __reduce_or_sync(0xffffffffu, flags);
        best = warp_max_u64(best);
        const bool bad_row = (flags & kPfBad) || !(ckey_val(best) > -kInf);
        const int am = ckey_idx(best);
        if (!kTree) {
            const bool pre = j.aux2 == kWalkPrefetched;
            const int kb = pre ? j.pad[0] : (A.k_per_req ? A.k_per_req[b] : A.K);
            if (bad_row) return greedy_finish(A, b, row, -1, st | 1);
            if (row == kb) return greedy_finish(A, b, row, am, st);
            const int y = pre ? j.y : A.draft[static_cast<long long>(b) * A.K + row];
            if (y < 0 || y >= A.V) st |= 8;
            if (y != am) return greedy_finish(A, b, row, am, st);
            Job nj = make_job(b, row + 1, 0, st);
            return nj;
        } else {
            const int acc = j.depth;
            if (bad_row) return tree_finish(A, b, acc, -1, st | 1);
            int child;
            if (sm.cb == b && sm.cnode == row && sm.cn >= 0) {
                // the cached children, ascending id: the first one carrying am
                uint32_t hit = 0;
                for (int c0 = 0; c0 < sm.cn && !hit; c0 += 32) {
                    const int c = c0 + l;
                    hit = __ballot_sync(0xffffffffu, c < sm.cn && sm.ctok[c] == am);
                    if (hit) child = sm.cid[c0 + __ffs(hit) - 1];
                }
                if (!hit) child = -1;
            } else {
                child = find_child_w(A.token, A.parent, A.num_nodes, A.N, b, row, am);
            }
            if (child < 0 || acc >= A.L) return tree_finish(A, b, acc, am, st);
            if (l == 0) {
                const int W = A.L + 1;
                A.out_tokens[static_cast<long long>(b) * W + acc] = am;
                A.path_nodes[static_cast<long long>(b) * W + acc + 1] = child;
            }
            __syncwarp();
            Job nj = make_job(b, child, 0, st);
            nj.depth = acc + 1;
            return nj;
        }
    }
};

template <class E, bool kTree>
__global__ void __launch_bounds__(kBlockThreads, 1) walk_kernel(const WalkArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    Engine<WalkOp<E, kTree>>::run(A, A.E.W, make_geo(A.E), smem);
}

template <class E, bool kTree>
static const void* walk_fn() { return reinterpret_cast<const void*>(&walk_kernel<E, kTree>); }

const void* walk_kernel_ptr(int ldt, int mode) {
    if (ldt == 0) return mode ? walk_fn<F32, true>() : walk_fn<F32, false>();
    return mode ? walk_fn<BF16, true>() : walk_fn<BF16, false>();
}

size_t walk_smem(int C, int own, int part_bytes, int stages, int chunk) {
    return Engine<WalkOp<F32, false>>::smem_bytes(C, own, part_bytes, stages, chunk);
}
int walk_part_bytes() { return static_cast<int>(sizeof(PartHdr)); }

}  // namespace spec

#ifdef SPEC_TRACE
// development builds: this translation unit's event trace buffer
extern "C" int spec_trace_setup_walk(void* buf, unsigned cap) {
    unsigned z = 0;
    if (cudaMemcpyToSymbol(spec::g_trace, &buf, sizeof(buf)) != cudaSuccess) return 1;
    if (cudaMemcpyToSymbol(spec::g_trace_cap, &cap, sizeof(cap)) != cudaSuccess) return 1;
    return cudaMemcpyToSymbol(spec::g_trace_n, &z, sizeof(z)) != cudaSuccess;
}
extern "C" unsigned spec_trace_count_walk(void) {
    unsigned n = 0;
    cudaMemcpyFromSymbol(&n, spec::g_trace_n, sizeof(n));
    return n;
}
#endif
