// spec_engine.cuh -- the persistent row-task engine shared by every
// verification kernel.
//
// Work model.  Every verification in this library walks, per request, a
// chain of vocabulary rows where row i+1 is read only if row i's decision
// says so (early exit).  A *task* is "process row r of request b"; it is cut
// into S contiguous *slices* of the vocabulary, and each (task, slice) pair
// is a *unit*.  A persistent grid of CTAs claims units from one global FIFO
// counter.  Inside a CTA a producer warp claims units and streams each
// unit's slice HBM -> shared memory with 1-D TMA bulk copies through a
// kStages mbarrier ring, while eight consumer warps process the chunks and
// write a small partial result per unit.  The CTA that completes the last slice of a task (atomic arrival
// counter, last-arriver pattern) combines the partials, takes the decision,
// and pushes the request's next task, if any, onto the queue.  Tasks of
// different requests and depths interleave freely: there is no grid-wide
// barrier, and a request's next row starts as soon as its decision is known.
//
// Waits.  A CTA that claimed a unit of a task not yet pushed waits for that
// task's ready flag, or for every request to be finished; the wait is
// bounded and gives up with SPEC_WS_ERR_WAIT.  Progress never depends on a
// waiting CTA: units are claimed in order and processed without waiting, so
// the kernel terminates even if only part of the grid is resident.
#pragma once

#include "spec_common.cuh"

namespace spec {

// Optional phase timers for development builds (-DSPEC_PROFILE): thread 0
// adds clock64() deltas per phase to g_prof[2*i] and counts to g_prof[2*i+1].
#ifdef SPEC_PROFILE
static __device__ unsigned long long g_prof[64];
#define SPEC_PROF_T(v) const long long v = clock64()
#define SPEC_PROF_ADD(i, v)                                                                   \
    do {                                                                                      \
        if (threadIdx.x == 0) {                                                               \
            atomicAdd(&g_prof[2 * (i)], static_cast<unsigned long long>(clock64() - (v)));    \
            atomicAdd(&g_prof[2 * (i) + 1], 1ull);                                            \
        }                                                                                     \
    } while (0)
#else
#define SPEC_PROF_T(v)
#define SPEC_PROF_ADD(i, v)
#endif

// Optional event trace for development builds (-DSPEC_TRACE): thread 0
// appends (globaltimer, SM, event, request, row, slice, aux) records to a
// buffer installed by the translation unit's spec_trace_setup_<name>().
#ifdef SPEC_TRACE
struct TraceRec {
    unsigned long long t;
    int sm, ev, b, row, slice, aux;
};
static __device__ TraceRec* g_trace;
static __device__ unsigned g_trace_cap;
static __device__ unsigned g_trace_n;
__device__ __forceinline__ void trace_ev(int ev, int b, int row, int slice, int aux) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    int sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    const unsigned i = atomicAdd(&g_trace_n, 1u);
    if (g_trace && i < g_trace_cap) {
        TraceRec r;
        r.t = t; r.sm = sm | (blockIdx.x << 8); r.ev = ev; r.b = b; r.row = row; r.slice = slice; r.aux = aux;
        g_trace[i] = r;
    }
}
#define SPEC_TRACE_EV(ev, b, row, slice, aux) \
    do { if (threadIdx.x == 0) ::spec::trace_ev((ev), (b), (row), (slice), (aux)); } while (0)
#define SPEC_TRACE_EXPORT(name)                                                              \
    extern "C" int spec_trace_setup_##name(void* buf, unsigned cap) {                        \
        unsigned z = 0;                                                                      \
        if (cudaMemcpyToSymbol(::spec::g_trace, &buf, sizeof(buf)) != cudaSuccess) return 1; \
        if (cudaMemcpyToSymbol(::spec::g_trace_cap, &cap, sizeof(cap)) != cudaSuccess) return 1; \
        return cudaMemcpyToSymbol(::spec::g_trace_n, &z, sizeof(z)) != cudaSuccess;          \
    }                                                                                        \
    extern "C" unsigned spec_trace_count_##name(void) {                                      \
        unsigned n = 0;                                                                      \
        cudaMemcpyFromSymbol(&n, ::spec::g_trace_n, sizeof(n));                               \
        return n;                                                                            \
    }
#else
#define SPEC_TRACE_EV(ev, b, row, slice, aux)
#define SPEC_TRACE_EXPORT(name)
#endif

// Ring geometry (development builds may override it).
#ifndef SPEC_CHUNK_BYTES
#define SPEC_CHUNK_BYTES 12288
#endif
#ifndef SPEC_STAGES
#define SPEC_STAGES 4
#endif
constexpr int kChunkBytes = SPEC_CHUNK_BYTES;   // one ring stage
constexpr int kStages = SPEC_STAGES;            // ring depth: 48 KiB in flight per CTA by default
static_assert(kChunkBytes % 4096 == 0 && kStages >= 2, "ring geometry");
constexpr int kMaxSlices = 32;

enum : uint32_t { kErrWait = 1u, kErrQueue = 2u };

// Queue control words, one 128-byte line per group so that the atomics on
// `head` and `tail` do not serialise with the polling of `done` / `error`.
struct Ctrl {
    uint32_t head;     // next unit index to claim
    uint32_t pad0[31];
    uint32_t tail;     // pushed tasks
    uint32_t pad1[31];
    uint32_t done;     // finished requests
    uint32_t error;    // kErr* bits
    uint32_t pad2[30];
    uint32_t hint0;    // top-k filter hint (value key) for first rows, from the latest finished row
    uint32_t pad3[31];
};
static_assert(sizeof(Ctrl) == 512, "Ctrl is four 128-byte lines");

struct Task {
    int32_t b, row, kind, aux;
};

struct ReqState {
    double m;          // row maximum (logit), carried to a residual pass
    double Z;          // normaliser, carried to a residual pass
    int32_t status;    // accumulated SPEC_ST_* bits
    int32_t pad0;
    double pad[5];
};
static_assert(sizeof(ReqState) == 64, "ReqState is 64 bytes");

// Slice partial written to global scratch; `keys` follow the header.
struct PartHdr {
    float vmax;        // slice maximum (over every element, NaN-propagating)
    int32_t cnt;       // number of keys written
    uint32_t flags;    // kPf* bits
    int32_t pad0;
    uint64_t kth;      // top-k: the slice's filter as a composite key / argmax: best key
    double sum;        // slice sum (meaning depends on the op)
    double sum2;
    float ly;          // chain: logit of the drafted token (slice holding it)
    float qy;          // chain: q of the drafted token (slice holding it)
    uint64_t pad1[2];
};
static_assert(sizeof(PartHdr) == 64, "PartHdr is 64 bytes");
enum : uint32_t { kPfBad = 1u, kPfOverflow = 2u, kPfHinted = 4u };

// Device view of the caller's workspace; offsets computed on the host.
struct Workspace {
    Ctrl* ctrl;
    uint32_t* ready;      // [maxt] ready flags of pushed tasks (zeroed per call)
    uint32_t* counter;    // [B] arrival counters (zeroed per call)
    Task* tasks;          // [maxt]
    ReqState* req;        // [B]
    unsigned char* part;  // [B][S] partials, part_stride bytes each
    unsigned char* extra; // [B] per-request op scratch, extra_stride bytes each
    uint32_t part_stride;
    uint32_t maxt;
    uint64_t extra_stride;
    int smax;             // partial slots per request
};

__device__ __forceinline__ PartHdr* part_hdr(const Workspace& W, int b, int s, int /*S*/) {
    return reinterpret_cast<PartHdr*>(W.part + (static_cast<size_t>(b) * W.smax + s) * W.part_stride);
}
__device__ __forceinline__ uint64_t* part_keys(const Workspace& W, int b, int s, int S) {
    return reinterpret_cast<uint64_t*>(part_hdr(W, b, s, S) + 1);
}

// ---------------------------------------------------------------------------
// queue
// ---------------------------------------------------------------------------
struct Claimed {
    Task task;
    int slice;
    int ok;
    uint32_t hint;     // a kernel-specific word the producer fetched with the claim
    int pad;
};

// The producer's claim of the next unit (one thread).  Units [0, B*S) are
// the initial tasks (kind = -1, row 0, one per request); unit u >= B*S
// belongs to pushed task (u/S - B), whose ready flag it waits for, bounded.
__device__ inline Claimed claim_unit(const Workspace& W, int B, int S) {
    Claimed c;
    c.ok = 1;
    c.hint = 0;
    c.pad = 0;
    const uint32_t u = atomicAdd(&W.ctrl->head, 1u);
    const uint32_t slot = u / static_cast<uint32_t>(S);
    c.slice = static_cast<int>(u % static_cast<uint32_t>(S));
    c.task.b = 0; c.task.row = 0; c.task.kind = -1; c.task.aux = 0;
    if (slot < static_cast<uint32_t>(B)) {
        c.task.b = static_cast<int>(slot);
        return c;
    }
    const uint32_t ti = slot - static_cast<uint32_t>(B);
    if (ti >= W.maxt) { c.ok = 0; return c; }
    uint32_t ns = 32;
    SPEC_TRACE_EV(10, -1, -1, -1, static_cast<int>(ti));
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire(&W.ready[ti])) {
            c.task.b = __ldcg(&W.tasks[ti].b);
            c.task.row = __ldcg(&W.tasks[ti].row);
            c.task.kind = __ldcg(&W.tasks[ti].kind);
            c.task.aux = __ldcg(&W.tasks[ti].aux);
            return c;
        }
        if (ld_acquire(&W.ctrl->done) >= static_cast<uint32_t>(B)) { c.ok = 0; return c; }
        if (ld_acquire(&W.ctrl->error) != 0) { c.ok = 0; return c; }   // another CTA gave up
        if (it >= kWaitLimit) { atomicOr(&W.ctrl->error, kErrWait); c.ok = 0; return c; }
        nanosleep_ns(ns);
        if (ns < 256) ns <<= 1;
    }
}

// Consumers: after the unit's partial is written.  Returns true (in every
// consumer thread) in the CTA that completed the task's last slice; that CTA
// owns the combine.
__device__ __forceinline__ bool arrive(const Workspace& W, int b, int S, int* sh) {
    csync();
    if (threadIdx.x == 0) {
        fence_acq_rel_gpu();   // release this CTA's partial
        const uint32_t prev = atomicAdd(&W.counter[b], 1u);
        int last = (prev == static_cast<uint32_t>(S - 1));
        if (last) {
            fence_acq_rel_gpu();   // acquire the other slices' partials
            W.counter[b] = 0;   // ready for the request's next task
        }
        *sh = last;
    }
    csync();
    return *sh != 0;
}

// Consumer thread 0 of the combining CTA: enqueue the request's next task.
__device__ __forceinline__ void push_task(const Workspace& W, Task t) {
    fence_acq_rel_gpu();
    const uint32_t ti = atomicAdd(&W.ctrl->tail, 1u);
    if (ti >= W.maxt) { atomicOr(&W.ctrl->error, kErrQueue); return; }
    __stcg(&W.tasks[ti].b, t.b);
    __stcg(&W.tasks[ti].row, t.row);
    __stcg(&W.tasks[ti].kind, t.kind);
    __stcg(&W.tasks[ti].aux, t.aux);
    st_release(&W.ready[ti], 1u);
}

// Consumer thread 0 of the combining CTA, after the request's outputs are
// written by all consumers (call after a csync()).
__device__ __forceinline__ void finish_request(const Workspace& W) {
    fence_acq_rel_gpu();
    atomicAdd(&W.ctrl->done, 1u);
}

// ---------------------------------------------------------------------------
// the producer / consumer pipeline of one CTA
// ---------------------------------------------------------------------------
// Warp kWarps (the producer) claims units, publishes each unit's descriptor
// through a two-slot queue, and streams the unit's chunks HBM -> shared
// memory with 1-D TMA bulk copies into a kStages ring.  The kWarps consumer
// warps take descriptors in order, wait for each chunk's `full` barrier,
// process it, and release the stage with one arrive per warp on its `empty`
// barrier; no consumer ever waits for another consumer while streaming.  The
// producer runs ahead by up to one unit, so a unit's claim and first bytes
// overlap the previous unit's tail, finish and combine.  Every wait is
// bounded; a timeout raises the CTA's abort flag and the workspace error.
struct Pipe {
    unsigned char* buf;    // kStages * kChunkBytes, 128-byte aligned
    uint64_t* full;        // [kStages] count 1: producer's expect_tx + the copies' bytes
    uint64_t* empty;       // [kStages] count kWarps: one arrive per consumer warp
    uint64_t* ufull;       // [2] count 1: descriptor published
    uint64_t* uempty;      // [2] count kWarps: descriptor read
    Claimed* desc;         // [2]
    volatile int* abort;   // a wait timed out in this CTA
    __device__ __forceinline__ unsigned char* slot(int s) const { return buf + s * kChunkBytes; }
};

// shared-memory control block of the pipe (part of every kernel's smem)
struct PipeSmem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t ufull[2];
    uint64_t uempty[2];
    Claimed desc[2];
    int abort;
    int pad[3];
};

// all kBlockThreads threads, once at kernel start
__device__ inline Pipe pipe_init(unsigned char* ring, PipeSmem& ps) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ps.full[s], 1);
            mbar_init(&ps.empty[s], kWarps);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&ps.ufull[j], 1);
            mbar_init(&ps.uempty[j], kWarps);
        }
        ps.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    Pipe P;
    P.buf = ring;
    P.full = ps.full; P.empty = ps.empty; P.ufull = ps.ufull; P.uempty = ps.uempty;
    P.desc = ps.desc;
    P.abort = &ps.abort;
    return P;
}

// What one unit streams: one row range (logits or q), or a logits range and
// the fp32 q range beside it in the same stages (the residual pass).
struct StreamPlan {
    const unsigned char* src0;   // element x0 of stream 0
    const unsigned char* src1;   // element x0 of stream 1 (fp32), or null
    int es0;                     // element bytes of stream 0
    int n;                       // elements
    int ce;                      // elements per chunk
    int nch;                     // chunks (0: the unit streams nothing)
};
__device__ __forceinline__ StreamPlan plan_none() {
    StreamPlan p;
    p.src0 = nullptr; p.src1 = nullptr; p.es0 = 4; p.n = 0; p.ce = 1; p.nch = 0;
    return p;
}
__device__ __forceinline__ StreamPlan plan_single(const void* row, int es, int x0, int x1) {
    StreamPlan p;
    p.src0 = static_cast<const unsigned char*>(row) + static_cast<long long>(x0) * es;
    p.src1 = nullptr;
    p.es0 = es;
    p.n = x1 > x0 ? x1 - x0 : 0;
    p.ce = kChunkBytes / es;
    p.nch = (p.n + p.ce - 1) / p.ce;
    return p;
}
template <int kEs>
__device__ __forceinline__ constexpr int dual_chunk_elems() { return (kChunkBytes / (kEs + 4)) & ~63; }
__device__ __forceinline__ StreamPlan plan_dual(const void* lrow, int es, const float* qrow, int x0, int x1) {
    StreamPlan p;
    p.src0 = static_cast<const unsigned char*>(lrow) + static_cast<long long>(x0) * es;
    p.src1 = reinterpret_cast<const unsigned char*>(qrow + x0);
    p.es0 = es;
    p.n = x1 > x0 ? x1 - x0 : 0;
    p.ce = es == 4 ? dual_chunk_elems<4>() : dual_chunk_elems<2>();
    p.nch = (p.n + p.ce - 1) / p.ce;
    return p;
}

// Producer lane: issue chunk c of plan p into stage s.  Bytes past the
// largest 16-byte multiple of each range are not copied (the consumers read
// them from global memory).
__device__ __forceinline__ void issue_chunk(const Pipe& P, const StreamPlan& p, int c, int s) {
    const int ne = min(p.ce, p.n - c * p.ce);
    const uint32_t b0 = static_cast<uint32_t>(ne * p.es0) & ~15u;
    const uint32_t b1 = p.src1 ? (static_cast<uint32_t>(ne * 4) & ~15u) : 0u;
    mbar_expect_tx(&P.full[s], b0 + b1);
    unsigned char* dst = P.slot(s);
    if (b0) tma_load_1d(dst, p.src0 + static_cast<long long>(c) * p.ce * p.es0, b0, &P.full[s]);
    if (b1) tma_load_1d(dst + p.ce * p.es0, p.src1 + static_cast<long long>(c) * p.ce * 4, b1, &P.full[s]);
}

// The producer warp's loop (lane 0 only).  `fetch(c)` may fill c.hint;
// `plan(c)` returns the unit's StreamPlan (tma: issue the chunks; otherwise
// the consumers copy them themselves).
template <class Fetch, class PlanF>
__device__ void producer_loop(const Workspace& W, int B, int S, const Pipe& P, bool tma, Fetch fetch, PlanF plan) {
    uint32_t seq = 0;          // chunks issued so far (ring sequence number)
    bool dead = false;
    for (uint32_t u = 0;; ++u) {
        const int j = u & 1;
        if (u >= 2 && !mbar_wait(&P.uempty[j], ((u >> 1) - 1) & 1u)) dead = true;
        Claimed c;
        if (dead || *P.abort) {
            c.ok = 0; c.slice = 0; c.hint = 0; c.pad = 0;
            c.task.b = 0; c.task.row = 0; c.task.kind = 0; c.task.aux = 0;
        } else {
            c = claim_unit(W, B, S);
            if (c.ok) fetch(c);
        }
        P.desc[j] = c;
        mbar_arrive(&P.ufull[j]);
        if (!c.ok) break;
        if (!tma) continue;
        const StreamPlan p = plan(c);
        for (int ci = 0; ci < p.nch; ++ci, ++seq) {
            const int s = static_cast<int>(seq % kStages);
            if (seq >= static_cast<uint32_t>(kStages) && !mbar_wait(&P.empty[s], ((seq / kStages) - 1) & 1u)) {
                dead = true;
                break;
            }
            if (*P.abort) { dead = true; break; }
            issue_chunk(P, p, ci, s);
        }
        if (dead) {
            // unblock consumers waiting for a descriptor, then stop
            *P.abort = 1;
            atomicOr(&W.ctrl->error, kErrWait);
        }
    }
    if (dead || *P.abort) {
        // wait (bounded) for the copies still in flight before the CTA can end
        const uint32_t first = seq > static_cast<uint32_t>(kStages) ? seq - kStages : 0u;
        for (uint32_t q = first; q < seq; ++q) mbar_wait(&P.full[q % kStages], (q / kStages) & 1u);
    }
}

// Consumers: the next unit's descriptor.  ok = 0 ends the consumer loop
// (every request finished, the queue closed, or an abort).
__device__ __forceinline__ Claimed next_unit(const Pipe& P, uint32_t u) {
    const int j = u & 1;
    const bool got = mbar_wait(&P.ufull[j], (u >> 1) & 1u);
    Claimed c = P.desc[j];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&P.uempty[j]);
    if (!got) *P.abort = 1;
    if (csync_or(!got || *P.abort)) c.ok = 0;
    return c;
}

// ---------------------------------------------------------------------------
// consumer side of a stream
// ---------------------------------------------------------------------------
// Calls, on every consumer thread, per chunk c:
//   fn.chunk_begin(c)                              -- chunk c is in shared memory
//   fn.pre_vec(active, vals, x) / fn.pre_scalar / fn.pre_end()
//                                                  -- chunk 0 only, if Fn::kPrepass
//                                                     and fn.use_prepass() (pre_end
//                                                     may csync())
//   fn.vec(active, vals, x)                        -- one 16-byte vector per thread and round
//   fn.scalar(active, v, x)                        -- tail elements that do not fill
//                                                     a vector, one per thread
//   fn.chunk_end(c, sm, cx0, nv)                   -- the chunk is still readable: sm
//                                                     holds nv full vectors from element cx0
//   fn.after_release(c)                            -- after the warp released the stage
// chunk_end and after_release run per warp (no consumer barrier).  Functors
// derive from FnHooks for the hooks they do not use.
struct FnHooks {
    static constexpr bool kPrepass = false;
    __device__ __forceinline__ bool use_prepass() const { return false; }
    template <int N> __device__ __forceinline__ void pre_vec(bool, const float (&)[N], int) {}
    __device__ __forceinline__ void pre_scalar(bool, float, int) {}
    __device__ __forceinline__ void pre_end() {}
    __device__ __forceinline__ void chunk_begin(int) {}
    __device__ __forceinline__ void chunk_end(int, const unsigned char*, int, int) {}
    __device__ __forceinline__ void after_release(int) {}
};

constexpr int kChunkVecs = kChunkBytes / 16;                  // vectors in a full chunk
constexpr int kFullRounds = (kChunkVecs + kThreads - 1) / kThreads;
static_assert(kChunkVecs % kThreads == 0, "a full chunk is a whole number of rounds");

// Wait for chunk `seq` (every consumer thread).  With tma = false the
// consumers copy it from global memory themselves (the producer issues
// nothing in that mode).
__device__ __forceinline__ bool take_chunk(const Pipe& P, uint32_t seq, bool tma, bool& dead,
                                           const StreamPlan& p, int c) {
    const int s = static_cast<int>(seq % kStages);
    if (tma) {
        const bool ok = !dead && mbar_wait(&P.full[s], (seq / kStages) & 1u);
        dead = !__all_sync(0xffffffffu, ok);   // warp-uniform from here on
        if (dead) *P.abort = 1;
        return !dead;
    }
    const int ne = min(p.ce, p.n - c * p.ce);
    unsigned char* sm = P.slot(s);
    csync();   // every consumer is done with this stage's previous chunk
    const unsigned char* g0 = p.src0 + static_cast<long long>(c) * p.ce * p.es0;
    if (p.es0 == 4) {
        for (int i = threadIdx.x; i < ne; i += kThreads)
            reinterpret_cast<uint32_t*>(sm)[i] = reinterpret_cast<const uint32_t*>(g0)[i];
    } else {
        for (int i = threadIdx.x; i < ne; i += kThreads)
            reinterpret_cast<uint16_t*>(sm)[i] = reinterpret_cast<const uint16_t*>(g0)[i];
    }
    if (p.src1) {
        const float* g1 = reinterpret_cast<const float*>(p.src1) + static_cast<long long>(c) * p.ce;
        float* d1 = reinterpret_cast<float*>(sm + p.ce * p.es0);
        for (int i = threadIdx.x; i < ne; i += kThreads) d1[i] = g1[i];
    }
    csync();
    return true;
}

// release chunk `seq` (per warp)
__device__ __forceinline__ void release_chunk(const Pipe& P, uint32_t seq, bool tma, bool dead) {
    if (!tma || dead) return;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&P.empty[seq % kStages]);
}

// Stream one row range (plan from plan_single) through fn.  Returns false
// (in every consumer thread) when a chunk wait timed out; the caller then
// leaves the kernel.  `seq` is the consumer's ring sequence number.
template <class E, class Fn>
__device__ bool consume_row(const Pipe& P, uint32_t& seq, const StreamPlan& p, bool tma, int x0, Fn& fn) {
    constexpr int VEC = E::kVec;
    bool dead = false;
    for (int c = 0; c < p.nch; ++c, ++seq) {
        const bool have = take_chunk(P, seq, tma, dead, p, c);
        const unsigned char* sm = P.slot(static_cast<int>(seq % kStages));
        const int ne = min(p.ce, p.n - c * p.ce);
        const int cx0 = x0 + c * p.ce;
        const int nv = (ne * E::kBytes) >> 4;
        const uint4* sv = reinterpret_cast<const uint4*>(sm);
        fn.chunk_begin(c);
        if (Fn::kPrepass && c == 0 && fn.use_prepass()) {
            for (int v = threadIdx.x; v < (have ? nv : 0); v += kThreads) {
                float vals[VEC];
                E::unpack(sv[v], vals);
                fn.pre_vec(true, vals, cx0 + v * VEC);
            }
            const int t0 = nv * VEC;
            if (have && t0 + static_cast<int>(threadIdx.x) < ne) {
                const int i = t0 + threadIdx.x;
                fn.pre_scalar(true, tma ? E::load(p.src0, static_cast<long long>(c) * p.ce + i) : E::load(sm, i),
                              cx0 + i);
            }
            fn.pre_end();
        }
        if (have) {
            if (nv == kChunkVecs) {
                // full chunk: every round's vector loaded first (independent loads)
                float vals[kFullRounds][VEC];
#pragma unroll
                for (int r = 0; r < kFullRounds; ++r) E::unpack(sv[r * kThreads + threadIdx.x], vals[r]);
#pragma unroll
                for (int r = 0; r < kFullRounds; ++r) fn.vec(true, vals[r], cx0 + (r * kThreads + threadIdx.x) * VEC);
            } else {
                const int rounds = (nv + kThreads - 1) / kThreads;
                for (int r = 0; r < rounds; ++r) {
                    const int v = r * kThreads + threadIdx.x;
                    float vals[VEC];
                    const bool act = v < nv;
                    if (act) E::unpack(sv[v], vals);
                    fn.vec(act, vals, cx0 + v * VEC);
                }
                const int t0 = nv * VEC;
                if (t0 < ne) {   // fewer than VEC elements left: at most one per thread
                    const int i = t0 + threadIdx.x;
                    const bool act = i < ne;
                    float v = 0.f;
                    if (act) v = tma ? E::load(p.src0, static_cast<long long>(c) * p.ce + i) : E::load(sm, i);
                    fn.scalar(act, v, cx0 + i);
                }
            }
            fn.chunk_end(c, sm, cx0, nv);
        }
        release_chunk(P, seq, tma, dead);
        if (have) fn.after_release(c);
    }
    return !csync_or(dead);
}

// Two ranges streamed together (plan from plan_dual): logits (E) and fp32 q
// over the same elements.  fn.vec2(active, lv[VEC], qv[VEC], x),
// fn.scalar2(active, l, q, x).
template <class E, class Fn>
__device__ bool consume_row2(const Pipe& P, uint32_t& seq, const StreamPlan& p, bool tma, int x0, Fn& fn) {
    constexpr int VEC = E::kVec;
    bool dead = false;
    for (int c = 0; c < p.nch; ++c, ++seq) {
        const bool have = take_chunk(P, seq, tma, dead, p, c);
        const unsigned char* sm = P.slot(static_cast<int>(seq % kStages));
        const int ne = min(p.ce, p.n - c * p.ce);
        const int cx0 = x0 + c * p.ce;
        const int qoff = p.ce * E::kBytes;
        if (have) {
            const int nv = ne / VEC;
            const int rounds = (nv + kThreads - 1) / kThreads;
            for (int r = 0; r < rounds; ++r) {
                const int v = r * kThreads + threadIdx.x;
                const bool act = v < nv;
                float lv[VEC], qv[VEC];
                if (act) {
                    E::unpack(reinterpret_cast<const uint4*>(sm)[v], lv);
                    const float4* q4 = reinterpret_cast<const float4*>(sm + qoff) + v * (VEC / 4);
#pragma unroll
                    for (int j = 0; j < VEC / 4; ++j) {
                        const float4 f = q4[j];
                        qv[4 * j] = f.x; qv[4 * j + 1] = f.y; qv[4 * j + 2] = f.z; qv[4 * j + 3] = f.w;
                    }
                }
                fn.vec2(act, lv, qv, cx0 + v * VEC);
            }
            const int t0 = nv * VEC;
            if (t0 < ne) {
                const int i = t0 + threadIdx.x;
                const bool act = i < ne;
                float l = 0.f, qq = 0.f;
                if (act) {
                    // bytes past the 16-byte-multiple prefix were not copied by TMA
                    const bool l_in = tma ? ((i * E::kBytes + E::kBytes) <= ((ne * E::kBytes) & ~15)) : true;
                    const bool q_in = tma ? ((i * 4 + 4) <= ((ne * 4) & ~15)) : true;
                    l = l_in ? E::load(sm, i) : E::load(p.src0, static_cast<long long>(c) * p.ce + i);
                    qq = q_in ? reinterpret_cast<const float*>(sm + qoff)[i]
                              : reinterpret_cast<const float*>(p.src1)[static_cast<long long>(c) * p.ce + i];
                }
                fn.scalar2(act, l, qq, cx0 + i);
            }
        }
        release_chunk(P, seq, tma, dead);
    }
    return !csync_or(dead);
}

// ---------------------------------------------------------------------------
// single-CTA passes over a global range (rescans and rare exact paths)
// ---------------------------------------------------------------------------

// Sum of w(x) over [x0, x1): fp32 per thread, fp64 across threads.
template <class W>
__device__ double cta_sum(int x0, int x1, W& w, double* red) {
    float acc = 0.f;
    for (int x = x0 + threadIdx.x; x < x1; x += kThreads) acc += w(x);
    return block_sum_d(static_cast<double>(acc), red);
}

// Inverse CDF over non-negative weights w(x), x ascending in [x0, x1): the
// smallest x with C(x) > t.  Blocks of kThreads*16 consecutive elements; each
// thread owns 16 consecutive elements (fp32 prefix inside, fp64 across), so
// every thread has 16 independent loads in flight per block.  If rounding
// leaves no crossing, returns the last x with w(x) > 0 (or x0).
template <class W>
__device__ int cta_icdf(int x0, int x1, double t, W& w, double* red, int* ired) {
    constexpr int PER = 16;
    double base = 0.0;
    int last_pos = -1;
    for (int b0 = x0; b0 < x1; b0 += kThreads * PER) {
        const int xs = b0 + threadIdx.x * PER;
        float wv[PER];
        float loc = 0.f;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int x = xs + j;
            wv[j] = (x < x1) ? w(x) : 0.f;
        }
        int lp = -1;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            loc += wv[j];
            if (wv[j] > 0.f) lp = xs + j;
        }
        double tot;
        const double ex = block_exscan_d(static_cast<double>(loc), red, tot);
        int found = 0x7fffffff;
        if (loc > 0.f && base + ex + static_cast<double>(loc) > t) {
            double c = base + ex;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                c += static_cast<double>(wv[j]);
                if (found == 0x7fffffff && wv[j] > 0.f && c > t) found = xs + j;
            }
        }
        csync();
        if (threadIdx.x == 0) { ired[0] = 0x7fffffff; ired[1] = -1; }
        csync();
        if (found != 0x7fffffff) atomicMin(&ired[0], found);
        if (lp >= 0) atomicMax(&ired[1], lp);
        csync();
        const int fb = ired[0];
        if (ired[1] > last_pos) last_pos = ired[1];
        csync();
        if (fb != 0x7fffffff) return fb;
        base += tot;
    }
    return last_pos >= 0 ? last_pos : x0;
}

// Every slice header of a task, in shared memory (loaded in parallel).
struct SliceHdrs {
    int cnt[kMaxSlices];
    int off[kMaxSlices + 1];     // exclusive prefix of cnt
    uint32_t flags[kMaxSlices];
    float vmax[kMaxSlices];
    uint64_t kth[kMaxSlices];
    double sum[kMaxSlices];
    double sum2[kMaxSlices];
    float ly[kMaxSlices];
    float qy[kMaxSlices];
};

__device__ inline void load_hdrs(const Workspace& W, int b, int S, SliceHdrs& H) {
    for (int s = threadIdx.x; s < S; s += kThreads) {
        const PartHdr* h = part_hdr(W, b, s, S);
        H.cnt[s] = __ldcg(&h->cnt);
        H.flags[s] = __ldcg(&h->flags);
        H.vmax[s] = __ldcg(&h->vmax);
        H.kth[s] = __ldcg(&h->kth);
        H.sum[s] = __ldcg(&h->sum);
        H.sum2[s] = __ldcg(&h->sum2);
        H.ly[s] = __ldcg(&h->ly);
        H.qy[s] = __ldcg(&h->qy);
    }
    csync();
    if (threadIdx.x == 0) {
        int a = 0;
        for (int s = 0; s < S; ++s) { H.off[s] = a; a += H.cnt[s]; }
        H.off[S] = a;
    }
    csync();
}

// Gather every slice key that `keep(key)` accepts into list[0..*lcnt)
// (order arbitrary); keys beyond `cap` set *oflow.  All loads independent.
template <class F>
__device__ inline void gather_keys(const Workspace& W, int b, int S, const SliceHdrs& H, F keep,
                                   uint64_t* list, int cap, int* lcnt, int* oflow) {
    if (threadIdx.x == 0) { *lcnt = 0; *oflow = 0; }
    csync();
    const int total = H.off[S];
    const int lane = threadIdx.x & 31;
    for (int f0 = 0; f0 < total; f0 += kThreads * 4) {
        uint64_t key[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = f0 + j * kThreads + threadIdx.x;
            key[j] = 0;
            if (f < total) {
                int s = 0;
                while (s + 1 < S && H.off[s + 1] <= f) ++s;
                key[j] = __ldcg(part_keys(W, b, s, S) + (f - H.off[s]));
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = f0 + j * kThreads + threadIdx.x;
            const bool p = f < total && keep(key[j]);
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            int base = 0;
            if (lane == 0 && bal) base = atomicAdd(lcnt, __popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (p) {
                const int pos = base + __popc(bal & ((1u << lane) - 1u));
                if (pos < cap) list[pos] = key[j];
                else *oflow = 1;
            }
        }
    }
    csync();
}

}  // namespace spec
