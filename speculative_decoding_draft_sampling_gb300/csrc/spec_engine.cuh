// spec_engine.cuh -- the cluster engine shared by every verification kernel.
//
// Work model.  Per request, a verification walks a chain of vocabulary rows
// in which row i+1 is read only when row i's decision says so (early exit).
// A thread-block cluster of C CTAs (one CTA per SM) owns up to R requests at
// a time, one per *slot*.  Every row is split across the cluster: CTA r
// streams elements [r*SL, min(V, (r+1)*SL)) of the row HBM -> shared memory
// with 1-D TMA bulk copies through a ring of mbarrier-tracked stages and
// reduces them to a small *partial*, which it stores into the shared memory
// of the slot's *leader* CTA (distributed shared memory) and counts on the
// leader's arrival mbarrier.  The leader's combiner warp takes the decision
// and posts the slot's next *job* (the request's next row, a residual pass,
// or the first row of a newly claimed request) to the mailbox of every CTA
// of the cluster.  Partials and jobs travel as asynchronous remote stores
// (st.async) whose bytes complete the receiving barrier's transaction count,
// so neither side pays a release fence at cluster scope.  Every CTA streams the jobs of all slots interleaved, so
// one slot's combine overlaps the other slots' streaming; slot s is led by
// CTA s mod C, so combines spread over the cluster.  Requests are claimed
// from one global counter whenever a slot frees up; there is no grid-wide
// barrier and no global queue.
//
// Roles inside a CTA (kBlockThreads threads):
//   warps 0..kWarps-1   consumers: take each job from the producer, process
//                       the streamed chunks, write the partial to the leader
//   warp kWarps         producer (lane 0): picks the next posted job of any
//                       slot (round robin), hands it to the consumers and
//                       issues its chunks
//   warp kWarps + 1     combiner: leads this CTA's slots (claims requests,
//                       combines their partials, posts their jobs)
//
// Waits.  Every wait is bounded (kMbarLimitNs of wall time); a wait that
// gives up sets the workspace error word and the CTA's abort flag, and every
// loop leaves.  No CTA leaves the kernel before the final cluster barrier,
// so no distributed-shared-memory store can target an exited CTA.
#pragma once

#include "spec_common.cuh"

namespace spec {

// Optional event trace for development builds (-DSPEC_TRACE): one lane
// appends (globaltimer, CTA, event, a, b, c) records to a buffer installed by
// the translation unit's spec_trace_setup_<name>() (every .cu file is its own
// device module with its own copy of the buffer pointer).
#ifdef SPEC_TRACE
struct TraceRec {
    unsigned long long t;
    int cta, ev, a, b, c, d;
};
static __device__ TraceRec* g_trace;
static __device__ unsigned g_trace_cap;
static __device__ unsigned g_trace_n;
static __device__ void trace_ev(int ev, int a, int b, int c);
#define SPEC_TRACE_EV(ev, a, b, c) ::spec::trace_ev((ev), (a), (b), (c))
#define SPEC_TRACE_T(v) const long long v = clock64()
#else
#define SPEC_TRACE_EV(ev, a, b, c)
#define SPEC_TRACE_T(v)
#endif

// Failure-path test builds (-DSPEC_TEST_HOOKS): when g_test_drop_post is
// set, the combiner of cluster rank 0 never posts its first slot's first job,
// so every wait that depends on it runs into its limit and the kernel must
// leave with the workspace error set.
#ifdef SPEC_TEST_HOOKS
static __device__ int g_test_drop_post;
#endif

// Ring geometry: the launch picks the stage size (a multiple of kChunkUnit:
// a full stage is whole groups of four rounds of 16-byte vectors) and how
// many stages fit, at most kStages.
constexpr int kStages = 8;
constexpr int kChunkUnit = 4 * 16 * (SPEC_THREADS);
constexpr int kChunkLarge = 2 * kChunkUnit;    // 48 KiB with 384 consumer threads
constexpr int kChunkSmall = kChunkUnit;        // 24 KiB

constexpr int kMaxC = 16;          // CTAs per cluster, at most
constexpr int kMaxSlots = 32;      // slots per cluster, at most
constexpr int kMaxOwn = 4;         // slots one CTA leads, at most
constexpr int kQ = 4;              // producer -> consumer job queue entries

enum : uint32_t { kErrWait = 1u, kErrQueue = 2u };
constexpr uint32_t kPersistTag = 0x5e1ec7edu;

// Workspace control block (caller memory; the first 128 bytes are zeroed
// by the call, the persist line is kept across calls).
struct Ctrl {
    uint32_t next;     // next request to claim
    uint32_t error;    // kErr* bits
    uint32_t pad0[30];
    uint32_t persist[32];   // [0] = kPersistTag when [1] holds a top-k filter hint for
                            // rows of vocabulary [2] and top-k [3]
};
static_assert(sizeof(Ctrl) == 256, "Ctrl is two 128-byte lines");

// A job: what the cluster does next for one slot.  Posted by the slot's
// leader into every CTA's mailbox; 64 bytes.
struct Job {
    int b;             // request; kJobStop: the slot retires
    int row;           // row index (meaning per kernel)
    int kind;          // per kernel
    int target;        // -1: every CTA streams its slice; else the one rank that works
    int st;            // the request's SPEC_ST_* bits so far
    uint32_t hint;     // per kernel (top-k filter hint, mask key)
    int aux, aux2;     // per kernel
    float f[4];        // per kernel
    int depth;         // tree walks: the depth of the node the job reads
    int y;             // chain: the row's drafted token when known (kYUnknown: not loaded yet)
    int pad[2];
};
static_assert(sizeof(Job) == 64, "Job is 64 bytes");
constexpr int kJobStop = -1;
constexpr int kJobDone = -2;       // returned by a combine: the request finished
constexpr int kYUnknown = -0x7fffffff;

__device__ __forceinline__ Job make_job(int b, int row, int kind, int st) {
    Job j;
    j.b = b; j.row = row; j.kind = kind; j.target = -1; j.st = st; j.hint = 0; j.aux = 0; j.aux2 = 0;
    j.f[0] = j.f[1] = j.f[2] = j.f[3] = 0.f;
    j.depth = 0; j.y = kYUnknown; j.pad[0] = j.pad[1] = 0;
    return j;
}
__device__ __forceinline__ Job job_done() { return make_job(kJobDone, 0, 0, 0); }

// Slice partial header (64 bytes); kernels append keys or bins after it.
struct PartHdr {
    float vmax;        // slice maximum (over every element, NaN-propagating)
    int32_t cnt;       // number of keys that follow
    uint32_t flags;    // kPf* bits
    int32_t tok;       // a token the slice found (argmax, a draw)
    uint64_t kth;      // top-k: the slice's filter as a composite key / argmax: best key
    float2 sum;        // slice sum, float-float (meaning per kernel)
    float2 sum2;
    float ly;          // chain: logit of the drafted token (slice holding it)
    float qy;          // chain: q of the drafted token (slice holding it)
    uint32_t hasy;     // 1: this slice holds the drafted token
    uint32_t pad1[3];
};
static_assert(sizeof(PartHdr) == 64, "PartHdr is 64 bytes");
enum : uint32_t { kPfBad = 1u, kPfOverflow = 2u, kPfHinted = 4u };

__device__ __forceinline__ const PartHdr* part_at(const unsigned char* parts, int pb, int r) {
    return reinterpret_cast<const PartHdr*>(parts + static_cast<size_t>(r) * pb);
}

// Device view of the caller's workspace.
struct Workspace {
    Ctrl* ctrl;
    unsigned char* extra;   // [B] per-request op scratch, extra_stride bytes each
    uint64_t extra_stride;
};

// Launch geometry every kernel's argument block carries (host-computed).
struct EngArgs {
    Workspace W;
    int stages;        // ring stages, 2..kStages
    int chunk;         // bytes of one stage, a multiple of kChunkUnit
    int C;             // CTAs per cluster (the launch's cluster size)
    int R;             // slots per cluster
    int SL;            // slice length in elements (a multiple of 64)
    int part_bytes;    // bytes of one partial (header + payload), multiple of 16
    int own;           // slots one CTA leads at most: ceil(R / C)
};

// cluster geometry of a launch, the same in every CTA but for the rank
struct Geo {
    int stages;        // ring stages
    int chunk;         // bytes of one stage
    int C;             // CTAs per cluster
    int R;             // slots per cluster
    int rank;          // this CTA's rank
    int SL;            // slice length in elements (a multiple of 64)
    int part_bytes;    // bytes of one partial slot (header + keys), multiple of 16
    int own;           // ceil(R / C)
};
__device__ __forceinline__ Geo make_geo(const EngArgs& E) {
    Geo g;
    g.C = static_cast<int>(cluster_size());
    g.rank = static_cast<int>(cluster_rank());
    g.R = E.R; g.SL = E.SL; g.part_bytes = E.part_bytes; g.own = E.own; g.stages = E.stages; g.chunk = E.chunk;
    return g;
}
__device__ __forceinline__ int slice_x0(const Geo& g, int r) { return r * g.SL; }
__device__ __forceinline__ int slice_x1(const Geo& g, int r, int V) { return min(V, (r + 1) * g.SL); }

// ---------------------------------------------------------------------------
// shared memory of the engine (every kernel's smem starts with the ring,
// then this block)
// ---------------------------------------------------------------------------
struct QEnt {
    Job job;
    int slot;
    int pad[3];
};
static_assert(sizeof(QEnt) == 80, "QEnt is 80 bytes");
struct EngSmem {
    uint64_t full[kStages];      // count 1: producer's expect_tx + the copies' bytes
    uint64_t empty[kStages];     // count kWarps: one arrive per consumer warp
    uint64_t qfull[kQ];          // count 1: producer posted a queue entry
    uint64_t qempty[kQ];         // count kWarps: every consumer warp read it
    uint64_t jfull[kMaxSlots];   // count 1: the slot's leader posted a job (remote arrive)
    uint64_t parr[kMaxOwn];      // count C: the partials of an own slot arrived (remote arrives)
    Job jd[kMaxSlots];           // mailboxes, written by the leaders
    Job cur[kMaxOwn];            // combiner: the job in flight of each own slot
    QEnt q[kQ];
    int abort;                   // a wait in this CTA gave up
    unsigned trace_n;            // development trace builds: this CTA's record count
    int pad[2];
};

#ifdef SPEC_TRACE
// every CTA appends to its own share of the buffer through a counter in its
// shared memory (no global atomic on the traced path); unused records stay
// zero.  The engine's shared block sits at the start of dynamic shared memory.
extern __shared__ __align__(128) unsigned char spec_trace_dyn[];
__device__ __forceinline__ void trace_reset_cta() { reinterpret_cast<EngSmem*>(spec_trace_dyn)->trace_n = 0; }
static __device__ void trace_ev(int ev, int a, int b, int c) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    const unsigned per = g_trace_cap / gridDim.x;
    const unsigned i = atomicAdd_block(&reinterpret_cast<EngSmem*>(spec_trace_dyn)->trace_n, 1u);
    if (g_trace && i < per) {
        TraceRec r;
        r.t = t; r.cta = blockIdx.x; r.ev = ev; r.a = a; r.b = b; r.c = c; r.d = 0;
        g_trace[static_cast<size_t>(blockIdx.x) * per + i] = r;
    }
}
#endif

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
// One try_wait on a phase parity: the hardware suspends the thread until the
// phase completes or kSuspendNs pass (a suspended warp issues nothing, so
// waiting warps leave the issue slots to the warps that work).
constexpr uint32_t kSuspendNs = 200000;
__device__ __forceinline__ bool mbar_try(const uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// the same for a phase completed by arrivals from other CTAs (acquire at
// cluster scope: their writes before the arrive are visible)
__device__ __forceinline__ bool mbar_try_cluster(const uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Wait for one mbarrier phase, up to kMbarLimitNs; gives up early when the
// CTA aborted or another CTA raised the workspace error.  false: gave up.
// The abort flag, the error word and the clock are looked at only every 64
// tries: a global load of the error word after every try would delay the
// next try by a memory round trip.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_phase(const uint64_t* bar, uint32_t parity, volatile int* abort,
                                           const Ctrl* ctrl) {
    if (kCluster ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    unsigned long long t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (kCluster ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort) return false;
            if (ld_relaxed(&ctrl->error) != 0u) return false;
            const unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kMbarLimitNs) return false;
        }
    }
}

// Poll test() (several barriers at once) until it holds, up to kMbarLimitNs:
// tight polling first, then a short sleep between polls.  false: gave up.
template <class T>
__device__ __forceinline__ bool poll_until(T test, volatile int* abort, const Ctrl* ctrl) {
    unsigned long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (test()) return true;
        if ((it & 255u) == 255u) {
            if (*abort) return false;
            if (ld_relaxed(&ctrl->error) != 0u) return false;
            const unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kMbarLimitNs) return false;
        }
        if (it >= 16u) nanosleep_ns(it >= 256u ? 128 : 32);
    }
}
__device__ __forceinline__ void raise_abort(volatile int* abort, Ctrl* ctrl) {
    *abort = 1;
    atomicOr(&ctrl->error, kErrWait);
}

// ---------------------------------------------------------------------------
// what a CTA streams for a job
// ---------------------------------------------------------------------------
// One row range (logits or q), or a logits range and the fp32 q range
// beside it in the same stages (the residual pass).
struct StreamPlan {
    const unsigned char* src0;   // element x0 of stream 0
    const unsigned char* src1;   // element x0 of stream 1 (fp32), or null
    int es0;                     // element bytes of stream 0
    int n;                       // elements
    int ce;                      // elements per chunk
    int nch;                     // chunks (0: the job streams nothing here)
};
__device__ __forceinline__ StreamPlan plan_none() {
    StreamPlan p;
    p.src0 = nullptr; p.src1 = nullptr; p.es0 = 4; p.n = 0; p.ce = 1; p.nch = 0;
    return p;
}
// `chunk`: the launch's stage size in bytes
__device__ __forceinline__ StreamPlan plan_single(const void* row, int es, int x0, int x1, int chunk) {
    StreamPlan p;
    p.src0 = static_cast<const unsigned char*>(row) + static_cast<long long>(x0) * es;
    p.src1 = nullptr;
    p.es0 = es;
    p.n = x1 > x0 ? x1 - x0 : 0;
    p.ce = chunk / es;
    p.nch = (p.n + p.ce - 1) / p.ce;
    return p;
}
__device__ __forceinline__ StreamPlan plan_dual(const void* lrow, int es, const float* qrow, int x0, int x1,
                                                int chunk) {
    StreamPlan p;
    p.src0 = static_cast<const unsigned char*>(lrow) + static_cast<long long>(x0) * es;
    p.src1 = reinterpret_cast<const unsigned char*>(qrow + x0);
    p.es0 = es;
    p.n = x1 > x0 ? x1 - x0 : 0;
    p.ce = (chunk / (es + 4)) & ~63;
    p.nch = (p.n + p.ce - 1) / p.ce;
    return p;
}

// The ring as the consumers and the producer see it.
struct Pipe {
    unsigned char* buf;    // stages * chunk bytes, 1024-byte aligned
    uint64_t* full;
    uint64_t* empty;
    volatile int* abort;
    Ctrl* ctrl;
    uint32_t stages;
    uint32_t magic;        // ceil(2^32 / stages): seq / stages by one multiply-high
    int chunk;             // bytes of one stage
    __device__ __forceinline__ unsigned char* slot(int s) const { return buf + s * chunk; }
    // ring position of sequence number seq: the stage, and how many times
    // the ring wrapped before it (exact for seq < 2^32 / stages)
    __device__ __forceinline__ int stage(uint32_t seq) const {
        return static_cast<int>(seq - __umulhi(seq, magic) * stages);
    }
    __device__ __forceinline__ uint32_t wraps(uint32_t seq) const { return __umulhi(seq, magic); }
};

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
    static constexpr bool kVec4 = false;   // the functor has vec4() for four rounds at once
    __device__ __forceinline__ bool use_prepass() const { return false; }
    template <int N> __device__ __forceinline__ void pre_vec(bool, const float (&)[N], int) {}
    __device__ __forceinline__ void pre_scalar(bool, float, int) {}
    __device__ __forceinline__ void pre_end() {}
    __device__ __forceinline__ void chunk_begin(int) {}
    __device__ __forceinline__ void chunk_end(int, const unsigned char*, int, int) {}
    __device__ __forceinline__ void after_release(int) {}
};

static_assert(kChunkUnit % (4 * 16 * kThreads) == 0, "a full stage is whole groups of four rounds");

// Plain-load mode (tma = false: pinned host memory read in place, or rows
// whose layout a bulk copy cannot take).  The consumers copy the chunks into
// the ring themselves with asynchronous 16-byte copies (global -> shared, no
// registers held), one chunk ahead: while a chunk is processed the next one
// is in flight, so a CTA keeps two chunks outstanding on the link.  Bytes
// past the last 16-byte multiple of a range, and ranges whose start is not
// 16-byte aligned, are copied element by element when their chunk is taken.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// the 16-byte part of n elements of es bytes at src, into dst (async)
__device__ __forceinline__ void copy_async(unsigned char* dst, const unsigned char* src, int n, int es) {
    if (reinterpret_cast<uintptr_t>(src) & 15u) return;
    const int nv = (n * es) >> 4;
    const uint32_t d = smem_u32(dst);
    for (int v = threadIdx.x; v < nv; v += kThreads) cp_async16(d + 16u * static_cast<uint32_t>(v), src + 16ll * v);
}
// the rest of it (everything when src is not 16-byte aligned), loaded now
__device__ __forceinline__ void copy_rest(unsigned char* dst, const unsigned char* src, int n, int es) {
    const int done = (reinterpret_cast<uintptr_t>(src) & 15u) ? 0 : (((n * es) >> 4) << 4) / es;
    if (es == 4) {
        for (int i = done + threadIdx.x; i < n; i += kThreads)
            reinterpret_cast<uint32_t*>(dst)[i] = __ldg(reinterpret_cast<const uint32_t*>(src) + i);
    } else {
        for (int i = done + threadIdx.x; i < n; i += kThreads)
            reinterpret_cast<uint16_t*>(dst)[i] = __ldg(reinterpret_cast<const unsigned short*>(src) + i);
    }
}
// chunk cc of plan p into dst, asynchronously; one commit group
__device__ __forceinline__ void chunk_async(const StreamPlan& p, int cc, unsigned char* dst) {
    const int nn = min(p.ce, p.n - cc * p.ce);
    copy_async(dst, p.src0 + static_cast<long long>(cc) * p.ce * p.es0, nn, p.es0);
    if (p.src1) copy_async(dst + p.ce * p.es0, p.src1 + static_cast<long long>(cc) * p.ce * 4, nn, 4);
    cp_async_commit();
}

// Wait for chunk `seq` (every consumer thread).  With tma = false the
// consumers copy it from global memory themselves (the producer issues
// nothing in that mode).
__device__ __forceinline__ bool take_chunk(const Pipe& P, uint32_t seq, bool tma, bool& dead,
                                           const StreamPlan& p, int c) {
    const int s = P.stage(seq);
    if (tma) {
        const uint32_t par = P.wraps(seq) & 1u;
        const bool ok = !dead && wait_phase(&P.full[s], par, P.abort, P.ctrl);
        dead = !__all_sync(0xffffffffu, ok);   // warp-uniform from here on
        if (dead) *P.abort = 1;
        return !dead;
    }
    const int ne = min(p.ce, p.n - c * p.ce);
    unsigned char* sm = P.slot(s);
    // every consumer is done with the chunks before this one, so this stage
    // and the next (the ring has at least two) are free
    csync();
    if (c == 0) chunk_async(p, 0, sm);
    const bool ahead = c + 1 < p.nch && P.stages >= 2;
    if (ahead) chunk_async(p, c + 1, P.slot(P.stage(seq + 1)));
    copy_rest(sm, p.src0 + static_cast<long long>(c) * p.ce * p.es0, ne, p.es0);
    if (p.src1) copy_rest(sm + p.ce * p.es0, p.src1 + static_cast<long long>(c) * p.ce * 4, ne, 4);
    if (ahead) cp_async_wait<1>();
    else cp_async_wait<0>();
    csync();
    return true;
}

// release chunk `seq` (per warp)
__device__ __forceinline__ void release_chunk(const Pipe& P, uint32_t seq, bool tma, bool dead) {
    if (!tma || dead) return;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&P.empty[P.stage(seq)]);
}

// Stream one row range (plan from plan_single) through fn.  Returns false
// (in every consumer thread) when a chunk wait gave up.  `seq` is the
// consumer's ring sequence number.
// The kRounds rounds of a full stage, four rounds' vectors loaded at a time
// (independent loads); functors with vec4() test the four together.
template <class E, int kRounds, class Fn>
__device__ __forceinline__ void full_stage(const uint4* sv, int cx0, Fn& fn) {
    constexpr int VEC = E::kVec;
    static_assert(kRounds % 4 == 0, "whole groups of four rounds");
#pragma unroll
    for (int g = 0; g < kRounds; g += 4) {
        float vals[4][VEC];
#pragma unroll
        for (int r = 0; r < 4; ++r) E::unpack(sv[(g + r) * kThreads + threadIdx.x], vals[r]);
        if constexpr (Fn::kVec4) {
            fn.vec4(vals, cx0 + (g * kThreads + threadIdx.x) * VEC);
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) fn.vec(true, vals[r], cx0 + ((g + r) * kThreads + threadIdx.x) * VEC);
        }
    }
}

template <class E, class Fn>
__device__ bool consume_row(const Pipe& P, uint32_t& seq, const StreamPlan& p, bool tma, int x0, Fn& fn) {
    constexpr int VEC = E::kVec;
    bool dead = false;
#ifdef SPEC_TRACE
    long long wait_cyc = 0, first_wait = 0, comp_cyc = 0, rel_cyc = 0;
    const long long t_beg = clock64();
#endif
    for (int c = 0; c < p.nch; ++c, ++seq) {
#ifdef SPEC_TRACE
        const long long tw = clock64();
#endif
        const bool have = take_chunk(P, seq, tma, dead, p, c);
#ifdef SPEC_TRACE
        wait_cyc += clock64() - tw;
        if (c == 0) first_wait = clock64() - tw;
        if (threadIdx.x == 0) SPEC_TRACE_EV(21, static_cast<int>(seq), static_cast<int>(clock64() - tw), c);
#endif
#ifdef SPEC_TRACE
        const long long tcb = clock64();
#endif
        const unsigned char* sm = P.slot(P.stage(seq));
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
            if (nv * 16 == P.chunk) {
                // full stage: whole groups of four rounds, unrolled
                if (P.chunk == kChunkLarge) full_stage<E, kChunkLarge / (16 * kThreads)>(sv, cx0, fn);
                else full_stage<E, kChunkSmall / (16 * kThreads)>(sv, cx0, fn);
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
#ifdef SPEC_TRACE
        const long long tce = clock64();
        comp_cyc += tce - tcb;
#endif
        release_chunk(P, seq, tma, dead);
        if (have) fn.after_release(c);
#ifdef SPEC_TRACE
        rel_cyc += clock64() - tce;
#endif
    }
#ifdef SPEC_TRACE
    if (threadIdx.x == 0) {
        SPEC_TRACE_EV(10, static_cast<int>(first_wait), static_cast<int>(wait_cyc), static_cast<int>(clock64() - t_beg));
        SPEC_TRACE_EV(13, static_cast<int>(comp_cyc), static_cast<int>(rel_cyc), p.nch);
    }
#endif
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
        const unsigned char* sm = P.slot(P.stage(seq));
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
// warp-level key selection over a shared-memory list (combiner warp)
// ---------------------------------------------------------------------------
// Keep list[i] with value key >= t, in place, order kept.
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
// the same on the full 64-bit key
__device__ inline int compact_key_w(uint64_t* list, int n, uint64_t t) {
    const int l = threadIdx.x & 31;
    const uint32_t lt = (1u << l) - 1u;
    int out = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + l;
        uint64_t key = 0;
        bool p = false;
        if (i < n) { key = list[i]; p = key >= t; }
        const uint32_t bal = __ballot_sync(0xffffffffu, p);
        if (p) list[out + __popc(bal & lt)] = key;
        out += __popc(bal);
    }
    __syncwarp();
    return out;
}

// The value key of the k-th largest key of list[0..n) (n >= k), by
// bisection over value keys (one warp reduction a step).
__device__ inline uint32_t kth_value_w(const uint64_t* list, int n, int k) {
    const int l = threadIdx.x & 31;
    uint32_t mx = 0, mn = 0xffffffffu;
    for (int i = l; i < n; i += 32) {
        const uint32_t h = static_cast<uint32_t>(list[i] >> 32);
        mx = max(mx, h);
        mn = min(mn, h);
    }
    uint32_t lo = warp_min_u32(mn), hi = warp_max_u32(mx);
    while (lo < hi) {
        const uint32_t mid = lo + static_cast<uint32_t>((static_cast<uint64_t>(hi) - lo + 1) >> 1);
        int c = 0;
        for (int i = l; i < n; i += 32) c += static_cast<uint32_t>(list[i] >> 32) >= mid;
        c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(c)));
        if (c >= k) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The largest composite key t with at least k keys of list[0..n) >= t (the
// exact k-th largest key; n >= k).
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

// ---------------------------------------------------------------------------
// the engine
// ---------------------------------------------------------------------------
// An Op provides (all device functions, every argument by const reference
// where it can):
//   using Args;  struct Smem (its own shared memory, after EngSmem)
//   int  R(A), ...                          (host side: see the kernel files)
//   Job  first(A, G, b, sm)                 combiner warp: the first job of
//                                           request b, or kJobDone when it
//                                           finishes without reading a row
//   StreamPlan plan(A, G, job)              producer: what this CTA streams
//   bool tma(A)                             TMA or plain loads
//   int  consume(A, G, P, seq, job, sm, out)   consumers: process this CTA's
//                                           part of the job, write the partial
//                                           (header + payload) to `out`; returns
//                                           its byte count (multiple of 16), or
//                                           -1 when a wait gave up
//   void prefetch(A, G, job, sm)            combiner warp, right after the job
//                                           was posted: load what its combine
//                                           will read into the combiner's own
//                                           copy of the job or its shared
//                                           memory (no-op allowed)
//   Job  combine(A, G, job, parts, sm)      combiner warp of the slot's leader:
//                                           parts = the C partials of the job;
//                                           returns the slot's next job, or
//                                           kJobDone when the request finished
template <class Op>
struct Engine {
    using Args = typename Op::Args;
    using OSmem = typename Op::Smem;

    // The combiner warp's copy of the arguments.  The combine steps are
    // separate (non-inlined) functions that reach the arguments through a
    // reference; a reference to the kernel's parameter block is a generic
    // pointer whose loads are slow (each a memory round trip, on the
    // critical path of every row), while one into shared memory is not.
    struct ArgsCopy {
        Args a;
        Workspace w;
        Geo g;
    };
    // dynamic shared memory: EngSmem | ArgsCopy | Op::Smem | partials (own
    // slots x C) | staging (one partial) | ring (stages x chunk bytes) |
    // kernel extras
    __host__ __device__ static size_t args_off() { return (sizeof(EngSmem) + 127) & ~size_t(127); }
    __host__ __device__ static size_t op_off() { return (args_off() + sizeof(ArgsCopy) + 127) & ~size_t(127); }
    __host__ __device__ static size_t part_off() { return (op_off() + sizeof(OSmem) + 127) & ~size_t(127); }
    __host__ __device__ static size_t stage_off(int C, int own, int part_bytes) {
        return part_off() + static_cast<size_t>(own) * C * part_bytes;
    }
    __host__ __device__ static size_t ring_off(int C, int own, int part_bytes) {
        return (stage_off(C, own, part_bytes) + part_bytes + 1023) & ~size_t(1023);
    }
    __host__ __device__ static size_t smem_bytes(int C, int own, int part_bytes, int stages, int chunk) {
        return ring_off(C, own, part_bytes) + static_cast<size_t>(stages) * chunk;
    }

    __device__ static void run(const Args& A, const Workspace& W, Geo G, unsigned char* smem) {
        EngSmem& es = *reinterpret_cast<EngSmem*>(smem);
        OSmem& os = *reinterpret_cast<OSmem*>(smem + op_off());
        unsigned char* parts = smem + part_off();
        unsigned char* stage = smem + stage_off(G.C, G.own, G.part_bytes);
        unsigned char* ring = smem + ring_off(G.C, G.own, G.part_bytes);
        const int C = G.C;
        if (threadIdx.x == 0) {
#ifdef SPEC_TRACE
            trace_reset_cta();
#endif
            for (int s = 0; s < G.stages; ++s) {
                mbar_init(&es.full[s], 1);
                mbar_init(&es.empty[s], kWarps);
            }
            for (int j = 0; j < kQ; ++j) {
                mbar_init(&es.qfull[j], 1);
                mbar_init(&es.qempty[j], kWarps);
            }
            for (int s = 0; s < kMaxSlots; ++s) mbar_init(&es.jfull[s], 1);
            for (int j = 0; j < kMaxOwn; ++j) mbar_init(&es.parr[j], C);
            es.abort = 0;
            fence_mbar_init();
        }
        Op::init_smem(A, G, os);
        ArgsCopy& ac = *reinterpret_cast<ArgsCopy*>(smem + args_off());
        static_assert(sizeof(Args) % 4 == 0 && sizeof(Workspace) % 4 == 0 && sizeof(Geo) % 4 == 0, "word copies");
        for (int i = threadIdx.x; i < static_cast<int>(sizeof(Args) / 4); i += blockDim.x)
            reinterpret_cast<uint32_t*>(&ac.a)[i] = reinterpret_cast<const uint32_t*>(&A)[i];
        if (threadIdx.x == 0) { ac.w = W; ac.g = G; }
        __syncthreads();
        // every CTA's barriers exist before any CTA posts to them
        cluster_sync();
        Pipe P;
        P.buf = ring; P.full = es.full; P.empty = es.empty; P.abort = &es.abort; P.ctrl = W.ctrl;
        P.stages = static_cast<uint32_t>(G.stages);
        P.magic = static_cast<uint32_t>(0xffffffffu / P.stages + 1u);
        P.chunk = G.chunk;
        const bool tma = Op::tma(A);
        if (threadIdx.x >= kCombiner0) {
            combiner(ac.a, ac.w, ac.g, es, os, parts);
        } else if (threadIdx.x >= kThreads) {
            if (threadIdx.x == kProducer) producer(A, W, G, es, P, tma);
        } else {
            consumers(A, W, G, es, os, P, tma, parts, stage);
        }
        __syncthreads();
        // no CTA leaves while another may still store to its shared memory
        cluster_sync();
    }

    // slots s with s % C == rank, s < R
    __device__ static int own_count(const Geo& G) { return G.rank < G.R ? (G.R - 1 - G.rank) / G.C + 1 : 0; }

    // ---- combiner warp: lead this CTA's slots -----------------------------
    __device__ static void post(const Geo& G, EngSmem& es, int s, const Job& j) {
        // lane r < C writes slot s's mailbox of CTA r and arrives on its jfull[s]
        const int l = threadIdx.x & 31;
        __syncwarp();
        if (l < G.C) {
            const uint32_t a = mapa(smem_u32(&es.jd[s]), static_cast<uint32_t>(l));
            const uint32_t bar = mapa(smem_u32(&es.jfull[s]), static_cast<uint32_t>(l));
            const uint4* v = reinterpret_cast<const uint4*>(&j);
            // the mailbox bytes are counted on the barrier as they land, so
            // the arrival needs no release fence (a release at cluster scope
            // would first wait for the outputs this warp just wrote to global
            // memory: about 1300 cycles)
            static_assert(sizeof(Job) == 64, "a job is four 16-byte stores");
            st_async_v4(a, v[0], bar);
            st_async_v4(a + 16, v[1], bar);
            st_async_v4(a + 32, v[2], bar);
            st_async_v4(a + 48, v[3], bar);
            mbar_arrive_expect_tx_cluster(bar, static_cast<uint32_t>(sizeof(Job)));
        }
        __syncwarp();
    }
    // Claim requests until one needs a row (or none are left: the stop job).
    // The first request of every slot is assigned, not claimed: slot s of
    // cluster c starts request s * clusters + c, so that a batch smaller
    // than the slot count spreads over the clusters one request each before
    // any cluster takes a second; later claims count on from there.
    __device__ static Job claim(const Args& A, const Workspace& W, const Geo& G, OSmem& os, int assigned = -1) {
        const int clusters = static_cast<int>(gridDim.x) / G.C;
        const int base = min(Op::batch(A), clusters * G.R);
        for (;;) {
            int b = assigned;
            assigned = -1;
            if (b < 0) {
                if ((threadIdx.x & 31) == 0) b = base + static_cast<int>(atomicAdd(&W.ctrl->next, 1u));
                b = __shfl_sync(0xffffffffu, b, 0);
            }
            Job j;
            if (b >= Op::batch(A)) return make_job(kJobStop, 0, 0, 0);
            j = Op::first(A, G, b, os);
            if (j.b != kJobDone) return j;
        }
    }
    __device__ static void combiner(const Args& A, const Workspace& W, const Geo& G, EngSmem& es, OSmem& os,
                                    unsigned char* parts) {
        const int nown = own_count(G);
        Job* cur = es.cur;      // shared memory: a register array indexed by slot would live in local memory
        uint32_t phase = 0;     // bit i: parity of own slot i's next arrival phase
        int active = 0;
        const int clusters = static_cast<int>(gridDim.x) / G.C;
        const int cl = static_cast<int>(cluster_id_x());
        for (int i = 0; i < nown; ++i) {
            const int s = G.rank + i * G.C;
            const int first_b = s * clusters + cl;
            const Job j = claim(A, W, G, os, first_b < Op::batch(A) ? first_b : -1);
            __syncwarp();
            if ((threadIdx.x & 31) == 0) cur[i] = j;
#ifdef SPEC_TEST_HOOKS
            if (!(g_test_drop_post && G.rank == 0 && i == 0 && blockIdx.x == 0))
#endif
            post(G, es, s, j);
            Op::prefetch(A, G, cur[i], os);
            if (j.b >= 0) active |= 1 << i;
        }
        while (active) {
            int ready = -1;
            bool ok;
            if (nown == 1) {
                ok = wait_phase<true>(&es.parr[0], phase & 1u, &es.abort, W.ctrl);
                ready = 0;
            } else {
                ok = poll_until([&]() {
                    for (int i = 0; i < nown; ++i)
                        if (((active >> i) & 1) && mbar_test_cluster(&es.parr[i], (phase >> i) & 1u)) {
                            ready = i;
                            return true;
                        }
                    return false;
                }, &es.abort, W.ctrl);
            }
            if (!__all_sync(0xffffffffu, ok)) { raise_abort(&es.abort, W.ctrl); break; }
            ready = __shfl_sync(0xffffffffu, ready, 0);
            const int i = ready;
            const int s = G.rank + i * G.C;
            phase ^= 1u << i;
            const unsigned char* pp = parts + static_cast<size_t>(i) * G.C * G.part_bytes;
            const Job cj = cur[i];
            if ((threadIdx.x & 31) == 0) SPEC_TRACE_EV(6, s, cj.b, cj.row);
            SPEC_TRACE_T(tk0);
            Job nx = Op::combine(A, G, cj, pp, os);
            SPEC_TRACE_T(tk1);
            if (nx.b == kJobDone) nx = claim(A, W, G, os);
            __syncwarp();
            if ((threadIdx.x & 31) == 0) cur[i] = nx;
            SPEC_TRACE_T(tk2);
            post(G, es, s, nx);
            Op::prefetch(A, G, cur[i], os);
            if ((threadIdx.x & 31) == 0) {
                SPEC_TRACE_EV(7, s, nx.b, nx.row);
                SPEC_TRACE_EV(14, static_cast<int>(tk1 - tk0), static_cast<int>(tk2 - tk1),
                              static_cast<int>(clock64() - tk2));
            }
            if (nx.b < 0) active &= ~(1 << i);
        }
    }

    // ---- producer lane ----------------------------------------------------
    __device__ static void producer(const Args& A, const Workspace& W, const Geo& G, EngSmem& es, const Pipe& P,
                                    bool tma) {
        uint32_t jph = 0;       // bit s: parity of slot s's next mailbox phase
        uint32_t seq = 0;       // chunks issued (ring sequence number)
        uint32_t qn = 0;        // queue entries posted
        int retired = 0, s0 = 0;
        bool dead = false;
        while (retired < G.R) {
            int s = -1;
            // of the posted jobs, the deepest row first (a request's rows are
            // sequential: its later rows are on the path that ends the call);
            // equal rows in round-robin order
            dead = !poll_until([&]() {
                int best_row = -1;
                for (int k = 0; k < G.R; ++k) {
                    const int t = (s0 + k) % G.R;
                    if (mbar_test_cluster(&es.jfull[t], (jph >> t) & 1u)) {
                        const int row = reinterpret_cast<const volatile Job*>(&es.jd[t])->row;
                        if (row > best_row) { best_row = row; s = t; }
                    }
                }
                return s >= 0;
            }, P.abort, W.ctrl);
            if (dead) break;
            s0 = s + 1 == G.R ? 0 : s + 1;
            jph ^= 1u << s;
            Job job;
            {
                const volatile Job* vj = &es.jd[s];
                job.b = vj->b; job.row = vj->row; job.kind = vj->kind; job.target = vj->target;
                job.st = vj->st; job.hint = vj->hint; job.aux = vj->aux; job.aux2 = vj->aux2;
                job.f[0] = vj->f[0]; job.f[1] = vj->f[1]; job.f[2] = vj->f[2]; job.f[3] = vj->f[3];
                job.depth = vj->depth; job.y = vj->y; job.pad[0] = job.pad[1] = 0;
            }
            if (job.b < 0) ++retired;
            // hand the job to the consumers
            const int qi = static_cast<int>(qn % kQ);
            if (qn >= static_cast<uint32_t>(kQ) && !wait_phase(&es.qempty[qi], ((qn / kQ) - 1) & 1u, P.abort, W.ctrl)) {
                dead = true;
                break;
            }
            es.q[qi].job = job;
            es.q[qi].slot = s;
            mbar_arrive(&es.qfull[qi]);
            ++qn;
            SPEC_TRACE_EV(1, s, job.b, job.row);
            if (job.b < 0 || !tma || (job.target >= 0 && job.target != G.rank)) continue;
            const StreamPlan p = Op::plan(A, G, job);
            for (int ci = 0; ci < p.nch; ++ci, ++seq) {
                const int st = P.stage(seq);
                if (seq >= P.stages && !wait_phase(&P.empty[st], (P.wraps(seq) - 1) & 1u, P.abort, W.ctrl)) {
                    dead = true;
                    break;
                }
                issue_chunk(P, p, ci, st);
                SPEC_TRACE_EV(20, static_cast<int>(seq), st, ci);
            }
            SPEC_TRACE_EV(2, s, job.b, job.row);
            if (dead) break;
        }
        if (dead) {
            raise_abort(P.abort, W.ctrl);
            // wait (bounded) for the copies still in flight before the CTA can end
            const uint32_t first = seq > P.stages ? seq - P.stages : 0u;
            for (uint32_t q = first; q < seq; ++q) {
                const int st = P.stage(q);
                const uint32_t par = P.wraps(q) & 1u;
                const unsigned long long t0 = globaltimer_ns();
                while (!mbar_test(&P.full[st], par) && globaltimer_ns() - t0 < kMbarLimitNs) nanosleep_ns(128);
            }
        }
    }

    // ---- consumer warps ---------------------------------------------------
    __device__ static void consumers(const Args& A, const Workspace& W, const Geo& G, EngSmem& es, OSmem& os,
                                     const Pipe& P, bool tma, unsigned char* parts, unsigned char* stage) {
        uint32_t seq = 0, qn = 0;
        int retired = 0;
        while (retired < G.R) {
            const int qi = static_cast<int>(qn % kQ);
            const bool ok = wait_phase(&es.qfull[qi], (qn / kQ) & 1u, P.abort, W.ctrl);
            if (csync_or(!ok)) { raise_abort(P.abort, W.ctrl); break; }
            const Job job = es.q[qi].job;
            const int s = es.q[qi].slot;
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(&es.qempty[qi]);
            ++qn;
            if (job.b < 0) { ++retired; continue; }
            const int leader = s % G.C;
            const int oi = s / G.C;
            const uint32_t arr = mapa(smem_u32(&es.parr[oi]), static_cast<uint32_t>(leader));
            if (job.target >= 0 && job.target != G.rank) {
                // not this CTA's job: acknowledge it (the leader posts the
                // slot's next job only after every CTA has taken this one)
                if (threadIdx.x == 0) mbar_arrive_expect_tx_cluster(arr, 0u);   // no bytes: relaxed suffices
                continue;
            }
            if (threadIdx.x == 0) SPEC_TRACE_EV(3, s, job.b, job.row);
            const int nb = Op::consume(A, G, P, seq, tma, job, os, stage);
            if (nb < 0) { raise_abort(P.abort, W.ctrl); break; }
            if (threadIdx.x == 0) SPEC_TRACE_EV(4, s, job.b, job.row);
            // the partial into the leader's slot area, then one counted arrival
            const uint32_t dst = mapa(smem_u32(parts + (static_cast<size_t>(oi) * G.C + G.rank) * G.part_bytes),
                                      static_cast<uint32_t>(leader));
            SPEC_TRACE_T(tx0);
            csync();   // the staging partial is complete
            SPEC_TRACE_T(tx1);
            // each 16 bytes counted on the leader's barrier as they land; the
            // barrier below only keeps the staging area until every thread
            // has read its share (the next job rewrites it)
            for (int i = threadIdx.x; i < nb / 16; i += kThreads)
                st_async_v4(dst + 16u * i, reinterpret_cast<const uint4*>(stage)[i], arr);
            csync();
            SPEC_TRACE_T(tx2);
            if (threadIdx.x == 0) {
                // one arrival that expects the partial's bytes: the phase
                // completes when every CTA has arrived and every byte landed
                mbar_arrive_expect_tx_cluster(arr, static_cast<uint32_t>(nb & ~15));
                SPEC_TRACE_EV(5, s, job.b, job.row);
                SPEC_TRACE_EV(26, static_cast<int>(tx1 - tx0), static_cast<int>(tx2 - tx1),
                              static_cast<int>(clock64() - tx2));
            }
        }
    }
};

}  // namespace spec
