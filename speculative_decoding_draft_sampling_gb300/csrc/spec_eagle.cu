// spec_eagle.cu -- EAGLE-2 dynamic draft tree: the grow step and the rerank.
//
// [SD-survey] = "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
// (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash, DDTree and
// DSpark), chzhyang.github.io, §4 "EAGLE-2": candidates grow along the
// branches of highest cumulative path confidence (the product of the draft
// probabilities along the path); every candidate is then reranked and the
// best form the tree to verify, whose depth and width follow the context.
//
// One expansion step is two launches: the engine reduces every frontier
// node's conditional draft row to its K2 most probable tokens (one unit per
// row, all rows of the step in parallel), then the grow kernel here -- one
// CTA per request -- appends the children to the request's node arrays and
// picks the next frontier: the Fn children of highest score, ties to the
// child appended first.  The rerank (one CTA per request) sorts every
// generated node by (score desc, depth asc, index asc) and keeps the root
// and the best budget - 1; a parent always sorts before its children (its
// score is no lower, its depth lower), so the kept set is a tree and is
// emitted parents first.  Both orders are strict and total (indices are
// distinct), so the grow places each child by its rank and the rerank sorts
// with a bitonic network over shared memory, both exactly.
#include "spec_chain.cuh"

namespace spec {

namespace {

constexpr int kGrowThreads = 256;
constexpr int kGrowMax = 2048;        // children of one step (F * K2)
constexpr int kRerankThreads = 512;
constexpr int kStTreeFull = 32;
constexpr int kStBadNode = 64;

struct SortEnt {
    unsigned long long s;   // order-preserving key of the score (larger first)
    int d;                  // depth (rerank) or 0 (grow)
    int i;                  // node index; 0x7fffffff: padding
};

// a double's order as an unsigned key (integer compares: the fp64 pipe is
// narrow on this part); -0 and +0 share a key
__device__ __forceinline__ unsigned long long score_key(double v) {
    unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(v));
    if ((b << 1) == 0ull) b = 0ull;
    return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

// the order both sorts use: real entries first; score desc; depth asc; index asc
__device__ __forceinline__ bool ent_first(const SortEnt& a, const SortEnt& b) {
    const bool va = a.i != 0x7fffffff, vb = b.i != 0x7fffffff;
    if (va != vb) return va;
    if (a.s != b.s) return a.s > b.s;
    if (a.d != b.d) return a.d < b.d;
    return a.i < b.i;
}

// Bitonic sort of e[0..n) (n a power of two) into ent_first order, all threads.
__device__ void bitonic_sort(SortEnt* e, int n) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const bool up = (i & k) == 0;
                    const SortEnt a = e[i], c = e[p];
                    if (up ? ent_first(c, a) : ent_first(a, c)) { e[i] = c; e[p] = a; }
                }
            }
            __syncthreads();
        }
    }
}

__host__ __device__ __forceinline__ int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

__global__ void __launch_bounds__(kGrowThreads) eagle_grow_kernel(const EagleGrowArgs A) {
    __shared__ int s_off[65], s_n[64], s_bad[64], s_node[64], s_dep[64];
    __shared__ double s_sc[64];
    __shared__ SortEnt s_ent[kGrowMax];
    __shared__ int s_st, s_g0, s_tot, s_ng;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int F = A.F, K2 = A.K2, G = A.G;
    auto hdr = [&](int f) {
        return reinterpret_cast<const EagleRowHdr*>(A.rows + static_cast<long long>(b * F + f) * A.row_stride);
    };
    // the row headers (each carries its frontier node, with the node's score
    // and depth), one thread each, and the generated count: one round of
    // independent loads; then the offsets on thread 0
    if (tid < F) {
        const EagleRowHdr* h = hdr(tid);
        s_n[tid] = h->n;
        s_bad[tid] = h->bad;
        s_node[tid] = h->node;
        s_dep[tid] = h->depth;
        s_sc[tid] = h->score;
    }
    if (tid == kGrowThreads - 1) s_ng = A.num_gen[b];
    __syncthreads();
    if (tid == 0) {
        int st = 0;
        int g0 = s_ng;
        if (g0 < 1 || g0 > G) { st |= kStBadNode; g0 = g0 < 1 ? 0 : G; }
        int off = 0;
        for (int f = 0; f < F; ++f) {
            const int n = s_n[f];
            s_off[f] = off;
            if (n == -2) st |= kStBadNode;
            if (n >= 0 && s_bad[f]) st |= 1;
            if (n > 0) off += n;
        }
        s_off[F] = off;
        if (off > G - g0) st |= kStTreeFull;
        s_st = st; s_g0 = g0; s_tot = off;
    }
    __syncthreads();
    const int g0 = s_g0, tot = s_tot;
    const int nc = tot < G - g0 ? tot : G - g0;   // children that fit, in (slot, rank) order
    for (int c = tid; c < nc; c += kGrowThreads) {
        int f = 0;
        while (s_off[f + 1] <= c) ++f;           // the slot whose children cover c
        const int r = c - s_off[f];
        const EagleRowHdr* h = hdr(f);
        const int* tok = reinterpret_cast<const int*>(h + 1);
        const float* prob = reinterpret_cast<const float*>(tok + K2);
        const long long nb = static_cast<long long>(b) * G;
        const double sc = s_sc[f] * static_cast<double>(prob[r]);
        const int g = g0 + c;
        A.token[nb + g] = tok[r];
        A.parent[nb + g] = s_node[f];
        A.depth[nb + g] = s_dep[f] + 1;
        A.score[nb + g] = sc;
        SortEnt e;
        e.s = score_key(sc); e.d = 0; e.i = g;
        s_ent[c] = e;
    }
    __syncthreads();
    // The next frontier: the Fn children first in that order, each placed
    // by its rank (how many children sort before it; the order is strict, the
    // indices being distinct).  One pass and no barrier: a sorting network
    // spent most of this kernel in its per-stage barriers.
    const int nn = A.Fn < nc ? A.Fn : nc;
    for (int c = tid; c < nc; c += kGrowThreads) {
        const SortEnt e = s_ent[c];
        int r = 0;
        for (int t = 0; t < nc; ++t) r += ent_first(s_ent[t], e) ? 1 : 0;
        if (r < nn) A.front_out[static_cast<long long>(b) * A.Fn + r] = e.i;
    }
    for (int j = nn + tid; j < A.Fn; j += kGrowThreads) A.front_out[static_cast<long long>(b) * A.Fn + j] = -1;
    if (tid == 0) {
        A.num_front_out[b] = nn;
        A.num_gen[b] = g0 + nc;
        A.status[b] = s_st;
    }
}

__global__ void __launch_bounds__(kRerankThreads) eagle_rerank_kernel(const EagleRerankArgs A, int P) {
    extern __shared__ __align__(16) unsigned char sm[];
    SortEnt* ent = reinterpret_cast<SortEnt*>(sm);                  // P entries
    int* pos = reinterpret_cast<int*>(ent + P);                     // G: sorted position + 1 of a node (0: none)
    int* nid = pos + A.G;                                           // G: emitted id of a node (-1: none)
    int* opar = nid + A.G;                                          // N: emitted parents
    __shared__ int s_st, s_g, s_cnt, s_bad;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int G = A.G, N = A.N, W = (N + 63) / 64;
    const long long nb = static_cast<long long>(b) * G, ob = static_cast<long long>(b) * N;
    if (tid == 0) {
        int st = 0, g = A.num_gen[b];
        if (g < 1 || g > G) { st |= kStBadNode; g = g < 1 ? 1 : G; }
        s_st = st; s_g = g; s_bad = 0;
    }
    __syncthreads();
    const int g = s_g;
    for (int i = tid; i < P; i += kRerankThreads) {
        SortEnt e;
        e.s = 0ull; e.d = 0; e.i = 0x7fffffff;
        if (i + 1 < g) { e.s = score_key(A.score[nb + i + 1]); e.d = A.depth[nb + i + 1]; e.i = i + 1; }
        ent[i] = e;
    }
    for (int i = tid; i < G; i += kRerankThreads) { pos[i] = 0; nid[i] = -1; }
    __syncthreads();
    bitonic_sort(ent, P);
    const int take = (N - 1) < (g - 1) ? (N - 1) : (g - 1);
    for (int k = tid; k < g - 1; k += kRerankThreads) pos[ent[k].i] = k + 1;
    __syncthreads();
    // kept entries whose parent is the root or a kept entry sorted earlier:
    // then the first `take` entries are the tree, in order
    for (int k = tid; k < take; k += kRerankThreads) {
        const int p = A.parent[nb + ent[k].i];
        const bool ok = p == 0 || (p > 0 && p < g && pos[p] > 0 && pos[p] - 1 < k);
        if (!ok) s_bad = 1;
    }
    __syncthreads();
    if (!s_bad) {
        for (int k = tid; k < take; k += kRerankThreads) nid[ent[k].i] = k + 1;
        if (tid == 0) { nid[0] = 0; s_cnt = take + 1; }
    } else if (tid == 0) {
        // a parent out of range or not kept: entries in order, each skipped
        // (and flagged) when its parent was not emitted before it
        nid[0] = 0;
        int cnt = 1;
        for (int k = 0; k < g - 1 && cnt < N; ++k) {
            const int i = ent[k].i;
            const int p = A.parent[nb + i];
            if (p < 0 || p >= g || nid[p] < 0) { s_st |= kStBadNode; continue; }
            nid[i] = cnt++;
        }
        s_cnt = cnt;
    }
    __syncthreads();
    const int cnt = s_cnt;
    // emitted node n <- its generated index (root: 0)
    if (tid == 0) {
        A.out_token[ob] = -1; A.out_parent[ob] = -1; A.out_depth[ob] = 0; A.out_score[ob] = 1.0;
        opar[0] = -1;
    }
    for (int k = tid; k < g - 1; k += kRerankThreads) {
        const int i = ent[k].i;
        const int n = nid[i];
        if (n > 0) {
            const int pe = nid[A.parent[nb + i]];
            A.out_token[ob + n] = A.token[nb + i];
            A.out_parent[ob + n] = pe;
            A.out_depth[ob + n] = A.depth[nb + i];
            A.out_score[ob + n] = A.score[nb + i];
            opar[n] = pe;
        }
    }
    for (int n = cnt + tid; n < N; n += kRerankThreads) {
        A.out_token[ob + n] = -1; A.out_parent[ob + n] = -1; A.out_depth[ob + n] = -1; A.out_score[ob + n] = 0.0;
    }
    __syncthreads();
    // ancestor masks: node n sees itself and its ancestors (each word built
    // in a register from the parent chain in shared memory, then stored once)
    for (int n = tid; n < N; n += kRerankThreads) {
        unsigned long long* mk = A.anc_mask + (ob + n) * W;
        for (int w = 0; w < W; ++w) {
            unsigned long long word = 0ull;
            if (n < cnt) {
                for (int m = n; m >= 0; m = opar[m])
                    if ((m >> 6) == w) word |= 1ull << (m & 63);
            }
            mk[w] = word;
        }
    }
    if (tid == 0) {
        A.num_nodes[b] = cnt;
        A.status[b] = s_st;
    }
}

size_t rerank_smem(int G, int N) {
    const int P = pow2_at_least(G > 2 ? G - 1 : 1);
    return static_cast<size_t>(P) * sizeof(SortEnt) + static_cast<size_t>(2 * G + N) * 4;
}

}  // namespace

cudaError_t eagle_grow_run(const EagleGrowArgs& A, cudaStream_t st) {
    eagle_grow_kernel<<<A.B, kGrowThreads, 0, st>>>(A);
    return cudaGetLastError();
}

cudaError_t eagle_rerank_run(const EagleRerankArgs& A, cudaStream_t st) {
    const int P = pow2_at_least(A.G > 2 ? A.G - 1 : 1);
    const size_t smem = rerank_smem(A.G, A.N);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(eagle_rerank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    eagle_rerank_kernel<<<A.B, kRerankThreads, smem, st>>>(A, P);
    return cudaGetLastError();
}

}  // namespace spec
