// spec_walk.cu -- argmax walks on the row-task engine.
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
#include "spec_chain.cuh"
#include "spec_select.cuh"

namespace spec {

struct __align__(16) WalkSmem {
    PipeSmem pipe;
    uint64_t red[kWarps];
    uint32_t wb[kWarps];
};

template <class E>
__device__ __forceinline__ const void* walk_row(const WalkArgs& A, int b, int i, bool tree) {
    long long r;
    if (!tree && A.k_per_req) r = static_cast<long long>(A.l_row_off[b] + i) * A.l_rs;
    else r = static_cast<long long>(b) * A.l_bs + static_cast<long long>(i) * A.l_rs;
    return static_cast<const unsigned char*>(A.logits) + r * E::kBytes;
}

// combiner warp
__device__ void greedy_finish(const WalkArgs& A, int b, int n, int last, int st) {
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
    if (l == 0) finish_request(A.W);
}

// combiner warp; path_nodes[b][0..acc] and out_tokens[b][0..acc-1] were
// written on the way
__device__ void tree_finish(const WalkArgs& A, int b, int acc, int last, int st) {
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
    if (l == 0) finish_request(A.W);
}

template <class E, bool kTree>
__device__ __forceinline__ bool walk_invalid(const WalkArgs& A, const Task& t) {
    if (kTree || t.kind >= 0) return false;
    const int kb = A.k_per_req ? A.k_per_req[t.b] : A.K;
    return kb < 0 || kb > A.K;
}

// The combine of one row (combiner warp): argmax over the slice partials,
// then the greedy decision or the tree step.
template <class E, bool kTree>
__device__ void walk_combine(const WalkArgs& A, const Job& job, uint32_t done, uint32_t base) {
    const int l = threadIdx.x & 31;
    const int b = job.task.b;
    const int row = job.task.row;
    const bool initial = job.task.kind < 0;
    const int acc = initial ? 0 : job.task.aux;
    int st = job.task.st;
    if (job.kind != 0) {   // invalid k
        greedy_finish(A, b, 0, -1, 16);
        return;
    }
    uint32_t flags = 0;
    uint64_t best = 0;
    const int S = task_S(A, job.task);
    for (int j = l; j < S; j += 32) {
        const PartHdr* h = part_hdr(A.W, b, j, S);
        flags |= __ldcg(&h->flags);
        const uint64_t k = __ldcg(&h->kth);
        best = k > best ? k : best;
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    best = warp_max_u64(best);
    const bool bad_row = (flags & kPfBad) || !(ckey_val(best) > -kInf);
    const int am = ckey_idx(best);
    if constexpr (!kTree) {
        const int kb = A.k_per_req ? A.k_per_req[b] : A.K;
        if (bad_row) { greedy_finish(A, b, row, -1, st | 1); return; }
        if (row == kb) { greedy_finish(A, b, row, am, st); return; }
        const int y = A.draft[static_cast<long long>(b) * A.K + row];
        if (y < 0 || y >= A.V) st |= 8;
        if (y != am) { greedy_finish(A, b, row, am, st); return; }
        if (l == 0) {
            Task nt;
            nt.b = b; nt.row = row + 1; nt.kind = 0; nt.aux = 0; nt.st = st; nt.base = base;
            int S1, SL1;
            pick_slices(A.B, A.V, A.S, A.S1, done, S1, SL1);
            push_task(A.W, nt, S1, SL1, false);
        }
    } else {
        if (bad_row) { tree_finish(A, b, acc, -1, st | 1); return; }
        // lowest child of `row` carrying the argmax token
        int child = 0x7fffffff;
        int nn = A.num_nodes[b];
        nn = nn < A.N ? nn : A.N;
        const int* par = A.parent + static_cast<long long>(b) * A.N;
        const int* tok = A.token + static_cast<long long>(b) * A.N;
        for (int c = l; c < nn; c += 32)
            if (par[c] == row && tok[c] == am) child = min(child, c);
        child = static_cast<int>(warp_min_u32(static_cast<uint32_t>(child)));
        if (child == 0x7fffffff || acc >= A.L) { tree_finish(A, b, acc, am, st); return; }
        if (l == 0) {
            const int W = A.L + 1;
            A.out_tokens[static_cast<long long>(b) * W + acc] = am;
            A.path_nodes[static_cast<long long>(b) * W + acc + 1] = child;
            Task nt;
            nt.b = b; nt.row = child; nt.kind = 0; nt.aux = acc + 1; nt.st = st; nt.base = base;
            int S1, SL1;
            pick_slices(A.B, A.V, A.S, A.S1, done, S1, SL1);
            push_task(A.W, nt, S1, SL1, false);   // outputs only: nothing for later tasks to read
        }
    }
}

template <class E, bool kTree>
__global__ void __launch_bounds__(kBlockThreads, kCtasPerSm) walk_kernel(const WalkArgs A) {
    extern __shared__ __align__(128) unsigned char smem[];
    auto& sh = *reinterpret_cast<WalkSmem*>(smem + kStages * kChunkBytes);
    const Pipe P = pipe_init(smem, sh.pipe);
    const bool tma = A.tma_l != 0;
    auto plan = [&](const Task& t, int slice) {
        if (walk_invalid<E, kTree>(A, t)) return plan_none();
        const int SL = task_SL(A, t);
        const int x0 = slice * SL, x1 = min(A.V, x0 + SL);
        return plan_single(walk_row<E>(A, t.b, t.row, kTree), E::kBytes, x0, x1);
    };
    if (threadIdx.x >= kCombiner0) {
        combiner_loop(P, [&](const Job& job) {
            uint32_t done;
            uint32_t base;
            if (comb_arrive(A.W, job.task, task_S(A, job.task), &done, &base)) walk_combine<E, kTree>(A, job, done, base);
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
        const bool invalid = walk_invalid<E, kTree>(A, t);
        PartHdr* ph = part_hdr(A.W, b, s, A.S);
        if (!invalid) {
            const int x0 = s * task_SL(A, t);
            ArgmaxFn<E> fn;
            if (!consume_row<E>(P, seq, plan(t, s), tma, x0, fn)) break;
            // per warp, then thread 0 over the warps (one barrier)
            const uint64_t wbest = warp_max_u64(fn.key());
            const uint32_t wbad = __reduce_or_sync(0xffffffffu, fn.bad_flag());
            if ((threadIdx.x & 31) == 0) { sh.red[threadIdx.x >> 5] = wbest; sh.wb[threadIdx.x >> 5] = wbad; }
            csync();
            if (threadIdx.x == 0) {
                uint64_t best = 0;
                uint32_t bad = 0;
                for (int j = 0; j < kWarps; ++j) { best = sh.red[j] > best ? sh.red[j] : best; bad |= sh.wb[j]; }
                ph->flags = bad ? kPfBad : 0u;
                ph->kth = best;
            }
        }
        csync();
        Job j;
        j.task = t; j.slice = s; j.kind = invalid ? 1 : 0; j.stop = 0; j.flags = 0;
        post_job(P, jseq, cseq, j, serve);
    }
    Job j;
    j.task.b = 0; j.task.row = 0; j.task.kind = 0; j.task.aux = 0; j.task.st = 0; j.task.base = 0;
    j.slice = 0; j.kind = 0; j.stop = 1; j.flags = 0;
    post_job(P, jseq, cseq, j, serve);
}

static size_t walk_smem() { return kStages * kChunkBytes + sizeof(WalkSmem); }

template <class E, bool kTree>
static cudaError_t walk_launch(const WalkArgs& A, int grid, cudaStream_t st) {
    const size_t smem = walk_smem();
    cudaError_t e = cudaFuncSetAttribute(walk_kernel<E, kTree>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    walk_kernel<E, kTree><<<grid, kBlockThreads, smem, st>>>(A);
    return cudaGetLastError();
}

template <class E, bool kTree>
static int walk_occ() {
    const int smem = static_cast<int>(walk_smem());
    int n = 0;
    cudaFuncSetAttribute(walk_kernel<E, kTree>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, walk_kernel<E, kTree>, kBlockThreads, smem);
    return n;
}

int walk_occupancy(int ldt, bool tree) {
    if (ldt == 0) return tree ? walk_occ<F32, true>() : walk_occ<F32, false>();
    return tree ? walk_occ<BF16, true>() : walk_occ<BF16, false>();
}

cudaError_t walk_run(const WalkArgs& A, bool tree, int grid, cudaStream_t st) {
    if (A.ldt == 0) return tree ? walk_launch<F32, true>(A, grid, st) : walk_launch<F32, false>(A, grid, st);
    return tree ? walk_launch<BF16, true>(A, grid, st) : walk_launch<BF16, false>(A, grid, st);
}

}  // namespace spec
