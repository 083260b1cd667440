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
// Waits.  A CTA that claimed a pushed unit not yet written waits for that
// unit's record (which carries the whole task), or for every request to be
// finished; the wait is bounded and gives up with SPEC_WS_ERR_WAIT.
// Progress never depends on a waiting CTA: units are claimed in order and
// processed without waiting, so the kernel terminates even if only part of
// the grid is resident.
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
#define SPEC_TRACE_EVW(ev, b, row, slice, aux) \
    do { if ((threadIdx.x & 31) == 0) ::spec::trace_ev((ev), (b), (row), (slice), (aux)); } while (0)
#define SPEC_TRACE_EV1(ev, b, row, slice, aux) ::spec::trace_ev((ev), (b), (row), (slice), (aux))
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
#define SPEC_TRACE_EVW(ev, b, row, slice, aux)
#define SPEC_TRACE_EV1(ev, b, row, slice, aux)
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
constexpr uint32_t kPersistTag = 0x5e1ec7edu;

// Queue control words, one 128-byte line per group so that the atomics on
// `head` and `tail` do not serialise with the polling of `done` / `error`.
struct Ctrl {
    uint32_t head;     // next initial unit to claim (the B*S0 units of the first rows)
    uint32_t pad0[31];
    uint32_t head1;    // next pushed unit to claim
    uint32_t pad4[31];
    unsigned long long tailc;   // (pushed tasks << 32) | pushed units
    uint32_t pad1[30];
    uint32_t done;     // finished requests
    uint32_t error;    // kErr* bits
    uint32_t pad2[30];
    uint32_t hint0;    // top-k filter hint (value key) for first rows, from the latest finished row
    uint32_t pad3[31];
};
static_assert(sizeof(Ctrl) == 640, "Ctrl is five 128-byte lines");

struct Task {
    int32_t b, row, kind, aux;
    int32_t st;       // the request's SPEC_ST_* bits so far
    uint32_t base;    // the request's arrival count before this task (mod 2^kBaseBits)
};
// A pushed task's kind word: bits 0-7 the kernel's kind, 8-13 its slice
// count, 14-31 its slice length / 64 (initial tasks have kind -1 and take
// the call's first-row slicing).
__host__ __device__ __forceinline__ int task_kind_base(int kind) { return kind & 0xff; }
__host__ __device__ __forceinline__ int task_kind_pack(int base, int S, int SL) {
    return (base & 0xff) | ((S & 63) << 8) | ((SL >> 6) << 14);
}
__host__ __device__ __forceinline__ int task_kind_S(int kind) { return (kind >> 8) & 63; }
__host__ __device__ __forceinline__ int task_kind_SL(int kind) { return ((kind >> 14) & 0x3ffff) << 6; }

struct ReqState {
    float m;           // row maximum (logit), carried to a residual pass
    float invZ;        // 1 / Z rounded to fp32: the residual pass and its rescan share it
    double pad[7];
};
static_assert(sizeof(ReqState) == 64, "ReqState is 64 bytes");

// Slice partial written to global scratch; `keys` follow the header.
struct PartHdr {
    float vmax;        // slice maximum (over every element, NaN-propagating)
    int32_t cnt;       // number of keys written
    uint32_t flags;    // kPf* bits
    int32_t pad0;
    uint64_t kth;      // top-k: the slice's filter as a composite key / argmax: best key
    float2 sum;        // slice sum, float-float (meaning depends on the op)
    float2 sum2;
    float ly;          // chain: logit of the drafted token (slice holding it)
    float qy;          // chain: q of the drafted token (slice holding it)
    uint64_t pad1[2];
};
static_assert(sizeof(PartHdr) == 64, "PartHdr is 64 bytes");
enum : uint32_t { kPfBad = 1u, kPfOverflow = 2u, kPfHinted = 4u };

// Device view of the caller's workspace; offsets computed on the host.
struct Workspace {
    Ctrl* ctrl;
    unsigned long long* urec;   // [maxu][2] pushed unit records, zero until pushed (zeroed per call)
    uint32_t* counter;    // [B] arrivals per request, never reset within a call (zeroed per call)
    ReqState* req;        // [B]
    unsigned char* part;  // [B][S] partials, part_stride bytes each
    unsigned char* extra; // [B] per-request op scratch, extra_stride bytes each
    uint32_t* persist;    // 128 bytes kept across calls on the same workspace (not zeroed):
                          // [0] = kPersistTag when [1] holds a top-k filter hint for rows
                          // of vocabulary [2] and top-k [3]
    uint32_t part_stride;
    uint32_t maxt;
    uint32_t maxu;
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
// A pushed unit's record carries its whole task, so that a claimer needs no
// further read and a push needs no fence when the task depends on nothing
// else the pusher wrote.  w0: b + 1 (bits 0-21), row (22-34), slice (35-40),
// st (41-45), base (46-62), and bit 63 when the push released earlier writes
// (the claimer then acquires); w1: the packed kind (low word), aux (high
// word).  Both words are nonzero once written (b + 1 >= 1; the kind word
// holds S >= 1).
constexpr int kBaseBits = 17;
constexpr unsigned long long kRecAcquire = 1ull << 63;
constexpr uint32_t kBaseMask = (1u << kBaseBits) - 1u;
constexpr int kMaxRecB = (1 << 22) - 2;     // requests per call
constexpr int kMaxRecRow = (1 << 13) - 1;   // row (or node) index
__device__ __forceinline__ void rec_encode(const Task& t, int slice, bool release, unsigned long long& w0,
                                           unsigned long long& w1) {
    w0 = static_cast<unsigned long long>(static_cast<uint32_t>(t.b + 1) & 0x3fffffu) |
         (static_cast<unsigned long long>(static_cast<uint32_t>(t.row) & 0x1fffu) << 22) |
         (static_cast<unsigned long long>(static_cast<uint32_t>(slice) & 63u) << 35) |
         (static_cast<unsigned long long>(static_cast<uint32_t>(t.st) & 31u) << 41) |
         (static_cast<unsigned long long>(t.base & kBaseMask) << 46) | (release ? kRecAcquire : 0ull);
    w1 = static_cast<unsigned long long>(static_cast<uint32_t>(t.kind)) |
         (static_cast<unsigned long long>(static_cast<uint32_t>(t.aux)) << 32);
}
__device__ __forceinline__ void rec_decode(unsigned long long w0, unsigned long long w1, Task& t, int& slice) {
    t.b = static_cast<int>(w0 & 0x3fffffu) - 1;
    t.row = static_cast<int>((w0 >> 22) & 0x1fffu);
    slice = static_cast<int>((w0 >> 35) & 63u);
    t.st = static_cast<int>((w0 >> 41) & 31u);
    t.base = static_cast<uint32_t>(w0 >> 46) & kBaseMask;
    t.kind = static_cast<int>(static_cast<uint32_t>(w1));
    t.aux = static_cast<int>(static_cast<uint32_t>(w1 >> 32));
}

struct Claimed {
    Task task;
    int slice;
    int ok;
    uint32_t hint;     // a kernel-specific word the producer fetched with the claim
    int pad;
};

// The producer's claim of the next unit (one thread).  First rows first
// (the initial units: row 0 of every request, S0 slices each): every
// request's chain starts as early as it can.  Then pushed tasks (rows that
// follow an accepted row, residual passes, retries) in push order, S1
// slices each; a claimer that finds none pushed yet takes the next pushed
// unit and waits (bounded) for its task, or for every request to finish.
// `cold` caches whether initial units may be left.
constexpr uint32_t kNoPre = 0xffffffffu;
__device__ inline Claimed claim_unit(const Workspace& W, int B, int S0, bool& cold, uint32_t& pre) {
    Claimed c;
    c.ok = 1;
    c.hint = 0;
    c.pad = 0;
    c.task.b = 0; c.task.row = 0; c.task.kind = -1; c.task.aux = 0; c.task.st = 0; c.task.base = 0;
    if (cold) {
        const uint32_t u0 = pre != kNoPre ? pre : atomicAdd(&W.ctrl->head, 1u);
        pre = kNoPre;
        if (u0 < static_cast<uint32_t>(B) * static_cast<uint32_t>(S0)) {
            c.slice = static_cast<int>(u0 % static_cast<uint32_t>(S0));
            c.task.b = static_cast<int>(u0 / static_cast<uint32_t>(S0));
            return c;
        }
        cold = false;
    }
    const uint32_t u = atomicAdd(&W.ctrl->head1, 1u);
    if (u >= W.maxu) { c.ok = 0; return c; }
    uint32_t ns = 32;
    SPEC_TRACE_EV(10, -1, -1, -1, static_cast<int>(u));
    for (uint32_t it = 0;; ++it) {
        // one round trip a poll: the record and the stop conditions together
        unsigned long long w0, w1;
        ld_relaxed_v2(W.urec + 2ull * u, w0, w1);
        const uint32_t fin = ld_relaxed(&W.ctrl->done);
        const uint32_t err = ld_relaxed(&W.ctrl->error);
        if (w0 != 0ull && w1 != 0ull) {
            if (w0 & kRecAcquire) fence_acq_rel_gpu();   // pairs with the pusher's release
            rec_decode(w0, w1, c.task, c.slice);
            return c;
        }
        if (fin >= static_cast<uint32_t>(B)) { c.ok = 0; return c; }
        if (err != 0) { c.ok = 0; return c; }   // another CTA gave up
        if (it >= kWaitLimit) { atomicOr(&W.ctrl->error, kErrWait); c.ok = 0; return c; }
        nanosleep_ns(ns);
        if (ns < 256) ns <<= 1;
    }
}

// Combiner warp: count the arrival of a finished unit (its partial was
// written by the consumers, ordered before the job hand-over).  Returns
// true in every lane when the unit completed the task's last slice; this
// CTA's combiner then owns the combine.  A request has one task in flight,
// and its counter only grows: the task's arrivals are those past its base,
// and the last one's count is the base of the request's next task.
__device__ __forceinline__ bool comb_arrive(const Workspace& W, const Task& t, int S, uint32_t* done_est,
                                            uint32_t* next_base) {
    int last = 0;
    uint32_t dn = 0, nb = 0;
    if ((threadIdx.x & 31) == 0) {
        fence_acq_rel_gpu();   // release the partial (cumulative over the hand-over)
        const uint32_t prev = atomicAdd(&W.counter[t.b], 1u);
        dn = ld_relaxed(&W.ctrl->done);   // (for the next row's slicing; not ordered)
        nb = (prev + 1u) & kBaseMask;
        last = (((prev + 1u - t.base) & kBaseMask) == static_cast<uint32_t>(S));
        if (last) fence_acq_rel_gpu();   // acquire the other slices' partials
    }
    if (done_est) *done_est = __shfl_sync(0xffffffffu, dn, 0);
    if (next_base) *next_base = __shfl_sync(0xffffffffu, nb, 0);
    return __shfl_sync(0xffffffffu, last, 0) != 0;
}

// One lane: enqueue the request's next task, cut into S slices of SL
// elements.  One 64-bit atomic reserves a task count (bounded by the
// workspace) and S unit records; each record carries the whole task.
__device__ __forceinline__ void push_task(const Workspace& W, Task t, int S, int SL, bool release) {
    t.kind = task_kind_pack(t.kind, S, SL);
    const unsigned long long r = atomicAdd(&W.ctrl->tailc, (1ull << 32) | static_cast<unsigned long long>(S));
    const uint32_t ti = static_cast<uint32_t>(r >> 32), u0 = static_cast<uint32_t>(r);
    if (ti >= W.maxt || u0 + static_cast<uint32_t>(S) > W.maxu) { atomicOr(&W.ctrl->error, kErrQueue); return; }
    // release: the task's units or combine read what the pusher wrote
    // before (request state beyond the record)
    if (release) fence_acq_rel_gpu();
    for (int s = 0; s < S; ++s) {
        unsigned long long w0, w1;
        rec_encode(t, s, release, w0, w1);
        st_relaxed_v2(W.urec + 2ull * (u0 + s), w0, w1);
    }
}

// Slices of a pushed row: a first row's while most requests are active;
// finer as requests finish, so that the remaining chains keep the grid busy
// (at most smax).  done = finished requests (an estimate).
#ifndef SPEC_SLICE_FACTOR
#define SPEC_SLICE_FACTOR 2   // pushed units per CTA when every active request has one row queued
#endif
__device__ __forceinline__ void pick_slices(int B, int V, int S0, int smax, uint32_t done, int& S, int& SL) {
    const int active = B - static_cast<int>(done) > 1 ? B - static_cast<int>(done) : 1;
    int s = (SPEC_SLICE_FACTOR * static_cast<int>(gridDim.x) + active - 1) / active;
    if (s < S0) s = S0;
    if (s > smax) s = smax;
    SL = (((V + s - 1) / s) + 63) & ~63;
    S = (V + SL - 1) / SL;
}

// Combiner lane 0, after the request's outputs are written by the warp.
// The count only tells claimers when to stop; the outputs are read after
// the kernel.
__device__ __forceinline__ void finish_request(const Workspace& W) {
    atomicAdd(&W.ctrl->done, 1u);
}

// ---------------------------------------------------------------------------
// the producer / consumer pipeline of one CTA
// ---------------------------------------------------------------------------
// A finished unit handed from the consumers to the combiner warp.
struct Job {
    Task task;       // as claimed (kind -1: an initial task)
    int slice;
    int kind;        // the unit's resolved kind
    int stop;        // no more jobs: the combiner leaves
    uint32_t flags;  // kernel-specific
};
constexpr int kJobs = 4;

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
    uint64_t* jfull;       // [kJobs] count 1: job posted by consumer thread 0
    uint64_t* jempty;      // [kJobs] count 1: job taken by the combiner
    Job* jobs;             // [kJobs]
    uint64_t* cready;
    uint64_t* cdone;
    volatile int* cflag;
    volatile int* abort;   // a wait timed out in this CTA
    __device__ __forceinline__ unsigned char* slot(int s) const { return buf + s * kChunkBytes; }
};

// shared-memory control block of the pipe (part of every kernel's smem)
struct PipeSmem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t ufull[2];
    uint64_t uempty[2];
    uint64_t jfull[kJobs];
    uint64_t jempty[kJobs];
    uint64_t cready;       // count 1: the combiner prepared a combine for the consumers
    uint64_t cdone;        // count 1: the consumers finished it
    Claimed desc[2];
    Job jobs[kJobs];
    int abort;
    int cflag;             // consumer thread 0's poll result, broadcast
    int pad[2];
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
        for (int j = 0; j < kJobs; ++j) {
            mbar_init(&ps.jfull[j], 1);
            mbar_init(&ps.jempty[j], 1);
        }
        mbar_init(&ps.cready, 1);
        mbar_init(&ps.cdone, 1);
        ps.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    Pipe P;
    P.buf = ring;
    P.full = ps.full; P.empty = ps.empty; P.ufull = ps.ufull; P.uempty = ps.uempty;
    P.desc = ps.desc;
    P.jfull = ps.jfull; P.jempty = ps.jempty; P.jobs = ps.jobs;
    P.cready = &ps.cready; P.cdone = &ps.cdone; P.cflag = &ps.cflag;
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
__device__ void producer_loop(const Workspace& W, int B, int S0, const Pipe& P, bool tma, Fetch fetch,
                              PlanF plan) {
    uint32_t seq = 0;          // chunks issued so far (ring sequence number)
    bool dead = false;
    bool cold = true;          // initial units may be left
    uint32_t pre = kNoPre;     // the next initial unit, taken while the current one streams
    for (uint32_t u = 0;; ++u) {
        const int j = u & 1;
        if (u >= 2 && !mbar_wait(&P.uempty[j], ((u >> 1) - 1) & 1u)) dead = true;
        Claimed c;
        if (dead || *P.abort) {
            c.ok = 0; c.slice = 0; c.hint = 0; c.pad = 0;
            c.task.b = 0; c.task.row = 0; c.task.kind = 0; c.task.aux = 0; c.task.st = 0; c.task.base = 0;
        } else {
            SPEC_TRACE_EV1(14, -1, -1, -1, static_cast<int>(u));
            c = claim_unit(W, B, S0, cold, pre);
            if (c.ok) fetch(c);
            SPEC_TRACE_EV1(13, c.task.b, c.task.row, c.slice, c.ok);
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
            // initial units are independent of every push: take the next one now,
            // its round trip overlaps this unit
            if (ci == 0 && cold && pre == kNoPre) pre = atomicAdd(&W.ctrl->head, 1u);
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

// Consumers (all threads): wait until thread 0's poll() reports done,
// serving the combines the combiner warp prepares meanwhile (serve() runs
// on every consumer thread; thread 0 then signals cdone).  `cseq` counts
// the combines served.  Every wait is bounded; false on a timeout or abort.
template <class Poll, class Serve>
__device__ bool consumer_wait(const Pipe& P, uint32_t& cseq, Poll poll, Serve serve) {
    unsigned long long t0 = 0;
    uint32_t ns = 0;
    for (uint32_t it = 0;; ++it) {
        if (threadIdx.x == 0) {
            int f = poll() ? 1 : 0;
            if (mbar_test(P.cready, cseq & 1u)) f |= 2;
            if (*P.abort) f |= 4;
            if ((it & 63u) == 63u) {
                const unsigned long long now = globaltimer_ns();
                if (t0 == 0) t0 = now;
                else if (now - t0 > kMbarLimitNs) f |= 4;
            }
            *P.cflag = f;
        }
        csync();
        const int f = *P.cflag;
        csync();   // every thread read the flag before thread 0 writes it again
        if (f & 2) {
            serve();
            csync();
            if (threadIdx.x == 0) mbar_arrive(P.cdone);
            ++cseq;
            ns = 0;
        }
        if (f & 1) return true;
        if (f & 4) { if (threadIdx.x == 0) *P.abort = 1; return false; }
        if (!(f & 2)) {
            if (ns) nanosleep_ns(ns);
            ns = ns ? (ns < 256 ? ns * 2 : ns) : 32;
        }
    }
}

// Combiner warp: hand the prepared combine number `cpub` to the consumers
// and go back to arrivals; the combine's shared memory stays theirs until
// combine_reuse().
__device__ inline void publish_combine(const Pipe& P, uint32_t& cpub) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(P.cready);
    ++cpub;
}

// Combiner warp: before writing the combine's shared memory again, wait
// (bounded) until the consumers finished the last published combine.
__device__ inline bool combine_reuse(const Pipe& P, uint32_t cpub) {
    if (cpub == 0) return true;
    if (*P.abort) return false;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(P.cdone, (cpub - 1) & 1u));
    if (!ok) *P.abort = 1;
    return ok;
}

// Consumers: the next unit's descriptor.  ok = 0 ends the consumer loop
// (every request finished, the queue closed, or an abort).
template <class Serve>
__device__ __forceinline__ Claimed next_unit(const Pipe& P, uint32_t u, uint32_t& cseq, Serve serve) {
    const int j = u & 1;
    const bool got = consumer_wait(P, cseq, [&]() { return mbar_test(&P.ufull[j], (u >> 1) & 1u); }, serve);
    Claimed c = P.desc[j];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&P.uempty[j]);
    if (!got || *P.abort) c.ok = 0;
    return c;
}

// Consumers (all threads): hand a finished unit (or the stop job) to the
// combiner warp, after a csync() that ordered every consumer's partial
// writes before it.  `jseq` counts the jobs posted so far.
template <class Serve>
__device__ inline void post_job(const Pipe& P, uint32_t& jseq, uint32_t& cseq, const Job& j, Serve serve) {
    const int s = static_cast<int>(jseq % kJobs);
    const uint32_t par = ((jseq / kJobs) - 1) & 1u;
    const bool ok = consumer_wait(P, cseq, [&]() {
        if (jseq >= static_cast<uint32_t>(kJobs) && !mbar_test(&P.jempty[s], par)) return false;
        P.jobs[s] = j;
        mbar_arrive(&P.jfull[s]);
        return true;
    }, serve);
    if (ok) ++jseq;
}

// The combiner warp's loop: take jobs in order until the stop job (or a
// timed-out wait).  on_job(job) runs on all 32 lanes; on_stop() runs before
// the stop job is marked taken (the consumers leave once it is), so that
// whatever the combiner handed them is finished first.
template <class F, class G>
__device__ void combiner_loop(const Pipe& P, F on_job, G on_stop) {
    for (uint32_t j = 0;; ++j) {
        const int s = static_cast<int>(j % kJobs);
        const bool got = __all_sync(0xffffffffu, mbar_wait(&P.jfull[s], (j / kJobs) & 1u));
        const Job job = P.jobs[s];
        if (got && job.stop) on_stop();
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&P.jempty[s]);
        if (!got) { *P.abort = 1; return; }
        if (job.stop) return;
        on_job(job);
    }
}
template <class F>
__device__ void combiner_loop(const Pipe& P, F on_job) {
    combiner_loop(P, on_job, []() {});
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
        if (c == 0) SPEC_TRACE_EV(15, -1, -1, -1, p.nch);
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

// Sum of w(x) over [x0, x1), float-float.
template <class W>
__device__ dfloat cta_sum(int x0, int x1, W& w, float2* red) {
    dfloat acc = df_make(0.f);
    for (int x = x0 + threadIdx.x; x < x1; x += kThreads) acc = df_add(acc, w(x));
    return block_sum_df(acc, red);
}

// Inverse CDF over non-negative weights w(x), x ascending in [x0, x1): the
// smallest x with C(x) > t.  Blocks of kThreads*16 consecutive elements; each
// thread owns 16 consecutive elements, so every thread has 16 independent
// loads in flight per block; prefixes in float-float.  If rounding leaves no
// crossing, returns the last x with w(x) > 0 (or x0).
template <class W>
__device__ int cta_icdf(int x0, int x1, dfloat t, W& w, float2* red, int* ired) {
    constexpr int PER = 16;
    dfloat base = df_make(0.f);
    int last_pos = -1;
    for (int b0 = x0; b0 < x1; b0 += kThreads * PER) {
        const int xs = b0 + threadIdx.x * PER;
        float wv[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int x = xs + j;
            wv[j] = (x < x1) ? w(x) : 0.f;
        }
        dfloat loc = df_make(0.f);
        int lp = -1;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            loc = df_add(loc, wv[j]);
            if (wv[j] > 0.f) lp = xs + j;
        }
        dfloat tot;
        const dfloat c0 = df_add(base, block_exscan_df(loc, red, tot));
        int found = 0x7fffffff;
        if (loc.hi > 0.f && df_gt(df_add(c0, loc), t)) {
            dfloat c = c0;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                c = df_add(c, wv[j]);
                if (found == 0x7fffffff && wv[j] > 0.f && df_gt(c, t)) found = xs + j;
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
        base = df_add(base, tot);
    }
    return last_pos >= 0 ? last_pos : x0;
}

// Every slice header of a task, in shared memory.
struct SliceHdrs {
    int cnt[kMaxSlices];
    int off[kMaxSlices + 1];     // exclusive prefix of cnt
    uint32_t flags[kMaxSlices];
    float vmax[kMaxSlices];
    uint64_t kth[kMaxSlices];
    float2 sum[kMaxSlices];
    float2 sum2[kMaxSlices];
    float ly[kMaxSlices];
    float qy[kMaxSlices];
};

// Combiner warp: lane s loads slice s's header (one round trip), offsets by
// a warp scan.  With `list`, the same round trip also fetches each slice's
// first keys into list[off_s ..] (speculatively: the slot always holds room
// for 2 * kPreKeys of them): kPreKeys per slice, or twice that when S <= 16
// (lane 16 + s fetches slice s's second kPreKeys).  Returns the keys per
// slice already in list (0 without list); gather_all_w fetches the rest.
constexpr int kPreKeys = 16;
__device__ inline int load_hdrs_w(const Workspace& W, int b, int S, SliceHdrs& H, uint64_t* list = nullptr,
                                  int cap = 0) {
    const int l = threadIdx.x & 31;
    const bool two = list && S <= 16;
    const int ps = two ? (l & 15) : l;              // the slice whose keys this lane fetches
    const int k0 = (two && l >= 16) ? kPreKeys : 0; // its first key
    const bool fetch = list && ps < S;
    int c = 0;
    ulonglong2 kp[kPreKeys / 2];
    if (fetch) {
        const ulonglong2* src = reinterpret_cast<const ulonglong2*>(part_keys(W, b, ps, S) + k0);   // 16-byte aligned
#pragma unroll
        for (int j = 0; j < kPreKeys / 2; ++j) kp[j] = __ldcg(src + j);
    }
    if (l < S) {
        const PartHdr* h = part_hdr(W, b, l, S);
        c = __ldcg(&h->cnt);
        H.cnt[l] = c;
        H.flags[l] = __ldcg(&h->flags);
        H.vmax[l] = __ldcg(&h->vmax);
        H.kth[l] = __ldcg(&h->kth);
        H.sum[l] = __ldcg(&h->sum);
        H.sum2[l] = __ldcg(&h->sum2);
        H.ly[l] = __ldcg(&h->ly);
        H.qy[l] = __ldcg(&h->qy);
    }
    int tot;
    const int off = warp_exscan_i(c, tot);
    if (l < S) H.off[l] = off;
    if (l == 0) H.off[S] = tot;
    const int cs = __shfl_sync(0xffffffffu, c, ps & 31);     // the fetched slice's count and offset
    const int os = __shfl_sync(0xffffffffu, off, ps & 31);
    if (fetch) {
#pragma unroll
        for (int j = 0; j < kPreKeys / 2; ++j) {
            const int a = k0 + 2 * j;
            if (a < cs && os + a < cap) list[os + a] = kp[j].x;
            if (a + 1 < cs && os + a + 1 < cap) list[os + a + 1] = kp[j].y;
        }
    }
    __syncwarp();
    return list ? (two ? 2 * kPreKeys : kPreKeys) : 0;
}

// Combiner warp: every slice key that keep(key) accepts into list[0..return)
// (order arbitrary); `oflow` when more than cap were accepted.  Each lane
// loads 8 keys per pass, all independent.
template <class F>
__device__ inline int gather_keys_w(const Workspace& W, int b, int S, const SliceHdrs& H, F keep,
                                    uint64_t* list, int cap, bool& oflow) {
    constexpr int U = 8;
    const int l = threadIdx.x & 31;
    const uint32_t lt = (1u << l) - 1u;
    const int total = H.off[S];
    int out = 0;
    int s = 0;   // slice of this lane's current key (its keys come in increasing order)
    for (int f0 = 0; f0 < total; f0 += 32 * U) {
        uint64_t key[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int f = f0 + j * 32 + l;
            key[j] = 0;
            if (f < total) {
                while (s + 1 < S && H.off[s + 1] <= f) ++s;
                key[j] = __ldcg(part_keys(W, b, s, S) + (f - H.off[s]));
            }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int f = f0 + j * 32 + l;
            const bool p = f < total && keep(key[j]);
            const uint32_t bal = __ballot_sync(0xffffffffu, p);
            if (p) {
                const int pos = out + __popc(bal & lt);
                if (pos < cap) list[pos] = key[j];
            }
            out += __popc(bal);
        }
    }
    oflow = out > cap;
    __syncwarp();
    return out < cap ? out : cap;
}

// Combiner warp: every key of every slice into list[H.off[s] ..] (lane s
// copies slice s; its loads are independent, 8 in flight).  Returns the
// count (at most cap; `oflow` when more).
__device__ inline int gather_all_w(const Workspace& W, int b, int S, const SliceHdrs& H, uint64_t* list,
                                   int cap, bool& oflow, int first = 0) {
    const int l = threadIdx.x & 31;
    const int total = H.off[S];
    oflow = total > cap;
    if (l < S) {
        const int c = H.cnt[l], o = H.off[l];
        const uint64_t* src = part_keys(W, b, l, S);
        for (int j0 = first; j0 < c; j0 += 8) {
            uint64_t key[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) key[j] = (j0 + j < c) ? __ldcg(src + j0 + j) : 0ull;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j0 + j < c && o + j0 + j < cap) list[o + j0 + j] = key[j];
        }
    }
    __syncwarp();
    return total < cap ? total : cap;
}

// Combiner warp: keep list[i] with value key >= t, in place, order kept.
__device__ inline int compact_w(uint64_t* list, int n, uint32_t t) {
    const int l = threadIdx.x & 31;
    const uint32_t lt = (1u << l) - 1u;
    int out = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + l;
        uint64_t key = 0;
        bool p = false;
        if (i < n) { key = list[i]; p = static_cast<uint32_t>(key >> 32) >= t; }
        const uint32_t bal = __ballot_sync(0xffffffffu, p);
        if (p) list[out + __popc(bal & lt)] = key;
        out += __popc(bal);
    }
    __syncwarp();
    return out;
}

// Combiner warp: the value key of the k-th largest key of list[0..n)
// (n >= k), by bisection over value keys (one warp reduction a step).
__device__ inline uint32_t kth_value_w(const uint64_t* list, int n, int k) {
    const int l = threadIdx.x & 31;
    uint32_t mx = 0;
    for (int i = l; i < n; i += 32) mx = max(mx, static_cast<uint32_t>(list[i] >> 32));
    uint32_t lo = 0, hi = warp_max_u32(mx);
    while (lo < hi) {
        const uint32_t mid = lo + static_cast<uint32_t>((static_cast<uint64_t>(hi) - lo + 1) >> 1);
        int c = 0;
        for (int i = l; i < n; i += 32) c += static_cast<uint32_t>(list[i] >> 32) >= mid;
        c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(c)));
        if (c >= k) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Combiner warp: the largest composite key t with at least k keys of
// list[0..n) >= t (the exact k-th largest key; n >= k).
__device__ inline uint64_t kth_key_w(const uint64_t* list, int n, int k) {
    const int l = threadIdx.x & 31;
    const uint32_t v = kth_value_w(list, n, k);
    uint64_t lo = static_cast<uint64_t>(v) << 32, hi = lo | 0xffffffffull;
    while (lo < hi) {
        const uint64_t d = hi - lo;
        const uint64_t mid = lo + (d >> 1) + (d & 1ull);
        int c = 0;
        for (int i = l; i < n; i += 32) c += list[i] >= mid;
        c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(c)));
        if (c >= k) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace spec
