// spec_engine.cuh -- the persistent row-task engine shared by every
// verification kernel.
//
// Work model.  Every verification in this library walks, per request, a
// chain of vocabulary rows where row i+1 is read only if row i's decision
// says so (early exit).  A *task* is "process row r of request b"; it is cut
// into S contiguous *slices* of the vocabulary, and each (task, slice) pair
// is a *unit*.  A persistent grid of CTAs claims units from one global FIFO
// counter; each unit streams its slice HBM -> shared memory with 1-D TMA
// bulk copies through a 4-stage mbarrier ring and writes a small partial
// result.  The CTA that completes the last slice of a task (atomic arrival
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

constexpr int kChunkBytes = 12288;   // one ring stage
constexpr int kStages = 4;           // ring depth: 48 KiB in flight per CTA
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
};

// Claim the next unit.  Units [0, B*S) are the initial tasks (kind = -1,
// row 0, one per request); unit u >= B*S belongs to pushed task (u/S - B).
__device__ __forceinline__ bool claim(const Workspace& W, int B, int S, Task& t, int& slice,
                                      Claimed* sh) {
    if (threadIdx.x == 0) {
        Claimed c;
        c.ok = 1;
        const uint32_t u = atomicAdd(&W.ctrl->head, 1u);
        const uint32_t slot = u / static_cast<uint32_t>(S);
        c.slice = static_cast<int>(u % static_cast<uint32_t>(S));
        if (slot < static_cast<uint32_t>(B)) {
            c.task.b = static_cast<int>(slot);
            c.task.row = 0;
            c.task.kind = -1;
            c.task.aux = 0;
        } else {
            const uint32_t ti = slot - static_cast<uint32_t>(B);
            if (ti >= W.maxt) {
                c.ok = 0;
            } else {
                uint32_t ns = 32;
                for (uint32_t it = 0;; ++it) {
                    if (ld_acquire(&W.ready[ti])) {
                        c.task.b = __ldcg(&W.tasks[ti].b);
                        c.task.row = __ldcg(&W.tasks[ti].row);
                        c.task.kind = __ldcg(&W.tasks[ti].kind);
                        c.task.aux = __ldcg(&W.tasks[ti].aux);
                        break;
                    }
                    if (ld_acquire(&W.ctrl->done) >= static_cast<uint32_t>(B)) { c.ok = 0; break; }
                    if (ld_acquire(&W.ctrl->error) != 0) { c.ok = 0; break; }   // another CTA gave up
                    if (it >= kWaitLimit) { atomicOr(&W.ctrl->error, kErrWait); c.ok = 0; break; }
                    nanosleep_ns(ns);
                    if (ns < 256) ns <<= 1;
                }
            }
        }
        *sh = c;
    }
    __syncthreads();
    const Claimed c = *sh;
    t = c.task;
    slice = c.slice;
    __syncthreads();
    return c.ok != 0;
}

// All threads: after the unit's partial is written.  Returns true in the CTA
// that completed the task's last slice; that CTA owns the combine.
__device__ __forceinline__ bool arrive(const Workspace& W, int b, int S, int* sh) {
    __syncthreads();
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
    __syncthreads();
    const int last = *sh;
    __syncthreads();
    return last != 0;
}

// Thread 0 of the combining CTA: enqueue the request's next task.
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

// Thread 0 of the combining CTA, after the request's outputs are written by
// the whole CTA (call after a __syncthreads()).
__device__ __forceinline__ void finish_request(const Workspace& W) {
    fence_acq_rel_gpu();
    atomicAdd(&W.ctrl->done, 1u);
}

// ---------------------------------------------------------------------------
// shared-memory ring fed by TMA bulk copies
// ---------------------------------------------------------------------------
struct Ring {
    unsigned char* buf;   // kStages * kChunkBytes, 128-byte aligned
    uint64_t* bar;        // kStages mbarriers
    uint32_t phase;       // bit s: parity of the next completion of stage s
    uint32_t err;

    __device__ void init(unsigned char* b, uint64_t* bars) {
        buf = b;
        bar = bars;
        phase = 0;
        err = 0;
        if (threadIdx.x == 0) {
            for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
            fence_mbar_init();
        }
        __syncthreads();
    }
    __device__ __forceinline__ unsigned char* slot(int s) const { return buf + s * kChunkBytes; }
    // thread 0: start the copies of one stage (sizes multiple of 16 bytes)
    __device__ __forceinline__ void issue(int s, const void* src0, uint32_t b0,
                                          const void* src1 = nullptr, uint32_t b1 = 0,
                                          uint32_t off1 = 0) {
        fence_proxy_async_smem();
        mbar_expect_tx(&bar[s], b0 + b1);
        if (b0) tma_load_1d(slot(s), src0, b0, &bar[s]);
        if (b1) tma_load_1d(slot(s) + off1, src1, b1, &bar[s]);
    }
    __device__ __forceinline__ void wait(int s) {
        if (!err && !mbar_wait(&bar[s], (phase >> s) & 1u)) err = 1;   // after one timeout, stop waiting
        phase ^= 1u << s;
    }
};

// Stream elements [x0, x1) of one row (16-byte aligned start when `tma`)
// through the ring.  Calls, on every thread, per chunk c:
//   fn.chunk_begin(c)                              -- chunk c is in shared memory
//   fn.pre_vec(active, vals, x) / fn.pre_scalar / fn.pre_end()
//                                                  -- chunk 0 only, if Fn::kPrepass
//                                                     and fn.use_prepass()
//   fn.vec(active, vals, x)                        -- one 16-byte vector per thread
//   fn.round_end()                                 -- after each round of vectors
//   fn.scalar(active, v, x)                        -- tail elements that do not fill
//                                                     a vector, one per thread
//   fn.chunk_end(c)                                -- before the CTA barrier that
//                                                     releases the stage
//   fn.after_release(c)                            -- after that barrier (uniform
//                                                     control flow: may synchronise)
// Functors derive from FnHooks for the hooks they do not use.
struct FnHooks {
    static constexpr bool kPrepass = false;
    __device__ __forceinline__ bool use_prepass() const { return false; }
    template <int N> __device__ __forceinline__ void pre_vec(bool, const float (&)[N], int) {}
    __device__ __forceinline__ void pre_scalar(bool, float, int) {}
    __device__ __forceinline__ void pre_end() {}
    __device__ __forceinline__ void chunk_begin(int) {}
    __device__ __forceinline__ void round_end() {}
    __device__ __forceinline__ void chunk_end(int) {}
    __device__ __forceinline__ void after_release(int) {}
};

template <class E, class Fn>
__device__ void stream_row(Ring& R, const void* row, bool tma, int x0, int x1, Fn& fn) {
    constexpr int CE = kChunkBytes / E::kBytes;
    constexpr int VEC = E::kVec;
    const int n = x1 - x0;
    if (n <= 0) return;
    const int nch = (n + CE - 1) / CE;
    const unsigned char* base = static_cast<const unsigned char*>(row) + static_cast<long long>(x0) * E::kBytes;
    if (tma && threadIdx.x == 0) {
        const int pre = nch < kStages ? nch : kStages;
        for (int c = 0; c < pre; ++c) {
            const int ne = min(CE, n - c * CE);
            R.issue(c, base + static_cast<long long>(c) * kChunkBytes, (ne * E::kBytes) & ~15);
        }
    }
    for (int c = 0; c < nch; ++c) {
        const int s = c % kStages;
        const int ne = min(CE, n - c * CE);
        const int cx0 = x0 + c * CE;
        unsigned char* sm = R.slot(s);
        if (tma) {
            R.wait(s);
        } else {
            const typename E::T* g = reinterpret_cast<const typename E::T*>(base) + static_cast<long long>(c) * CE;
            typename E::T* d = reinterpret_cast<typename E::T*>(sm);
            for (int i = threadIdx.x; i < ne; i += kThreads) d[i] = g[i];
            __syncthreads();
        }
        const int nv = (ne * E::kBytes) >> 4;
        const int rounds = (nv + kThreads - 1) / kThreads;
        fn.chunk_begin(c);
        if (Fn::kPrepass && c == 0 && fn.use_prepass()) {
            for (int r = 0; r < rounds; ++r) {
                const int v = r * kThreads + threadIdx.x;
                float vals[VEC];
                const bool act = v < nv;
                if (act) E::unpack(reinterpret_cast<const uint4*>(sm)[v], vals);
                fn.pre_vec(act, vals, cx0 + v * VEC);
            }
            const int t0 = (nv << 4) / E::kBytes;
            if (t0 < ne) {
                const int i = t0 + threadIdx.x;
                const bool act = i < ne;
                float v = 0.f;
                if (act) v = tma ? E::load(base, static_cast<long long>(c) * CE + i)
                                 : E::load(sm, i);
                fn.pre_scalar(act, v, cx0 + i);
            }
            fn.pre_end();
        }
        for (int r = 0; r < rounds; ++r) {
            const int v = r * kThreads + threadIdx.x;
            float vals[VEC];
            const bool act = v < nv;
            if (act) E::unpack(reinterpret_cast<const uint4*>(sm)[v], vals);
            fn.vec(act, vals, cx0 + v * VEC);
            fn.round_end();
        }
        const int t0 = (nv << 4) / E::kBytes;
        if (t0 < ne) {   // fewer than VEC elements left: at most one per thread
            const int i = t0 + threadIdx.x;
            const bool act = i < ne;
            float v = 0.f;
            if (act) v = tma ? E::load(base, static_cast<long long>(c) * CE + i) : E::load(sm, i);
            fn.scalar(act, v, cx0 + i);
            fn.round_end();
        }
        fn.chunk_end(c);
        __syncthreads();   // every thread is done with stage s
        if (tma && threadIdx.x == 0 && c + kStages < nch) {
            const int c2 = c + kStages;
            const int ne2 = min(CE, n - c2 * CE);
            R.issue(s, base + static_cast<long long>(c2) * kChunkBytes, (ne2 * E::kBytes) & ~15);
        }
        fn.after_release(c);
    }
}

// Two rows streamed together: logits (E) and fp32 q over the same element
// range.  fn.vec2(active, lv[VEC], qv[VEC], x), fn.scalar2(active, l, q, x).
template <class E, class Fn>
__device__ void stream_row2(Ring& R, const void* lrow, const float* qrow, bool tma,
                            int x0, int x1, Fn& fn) {
    constexpr int CE = (kChunkBytes / (E::kBytes + 4)) & ~63;
    constexpr int VEC = E::kVec;
    constexpr int LOFF = 0;
    constexpr int QOFF = CE * E::kBytes;
    const int n = x1 - x0;
    if (n <= 0) return;
    const int nch = (n + CE - 1) / CE;
    const unsigned char* lb = static_cast<const unsigned char*>(lrow) + static_cast<long long>(x0) * E::kBytes;
    const float* qb = qrow + x0;
    auto issue = [&](int c, int s) {
        const int ne = min(CE, n - c * CE);
        R.issue(s, lb + static_cast<long long>(c) * CE * E::kBytes, (ne * E::kBytes) & ~15,
                qb + static_cast<long long>(c) * CE, (ne * 4) & ~15, QOFF);
    };
    if (tma && threadIdx.x == 0) {
        const int pre = nch < kStages ? nch : kStages;
        for (int c = 0; c < pre; ++c) issue(c, c);
    }
    for (int c = 0; c < nch; ++c) {
        const int s = c % kStages;
        const int ne = min(CE, n - c * CE);
        const int cx0 = x0 + c * CE;
        unsigned char* sm = R.slot(s);
        if (tma) {
            R.wait(s);
        } else {
            const typename E::T* g = reinterpret_cast<const typename E::T*>(lb) + static_cast<long long>(c) * CE;
            typename E::T* d = reinterpret_cast<typename E::T*>(sm + LOFF);
            float* dq = reinterpret_cast<float*>(sm + QOFF);
            for (int i = threadIdx.x; i < ne; i += kThreads) {
                d[i] = g[i];
                dq[i] = qb[static_cast<long long>(c) * CE + i];
            }
            __syncthreads();
        }
        // vectors of VEC logits (16 bytes) and VEC q values (VEC*4 bytes)
        const int nv = ne / VEC;
        const int rounds = (nv + kThreads - 1) / kThreads;
        for (int r = 0; r < rounds; ++r) {
            const int v = r * kThreads + threadIdx.x;
            const bool act = v < nv;
            float lv[VEC], qv[VEC];
            if (act) {
                E::unpack(reinterpret_cast<const uint4*>(sm + LOFF)[v], lv);
                const float4* q4 = reinterpret_cast<const float4*>(sm + QOFF) + v * (VEC / 4);
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
                l = l_in ? E::load(sm + LOFF, i) : E::load(lb, static_cast<long long>(c) * CE + i);
                qq = q_in ? reinterpret_cast<const float*>(sm + QOFF)[i] : qb[static_cast<long long>(c) * CE + i];
            }
            fn.scalar2(act, l, qq, cx0 + i);
        }
        __syncthreads();
        if (tma && threadIdx.x == 0 && c + kStages < nch) issue(c + kStages, s);
    }
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
        __syncthreads();
        if (threadIdx.x == 0) { ired[0] = 0x7fffffff; ired[1] = -1; }
        __syncthreads();
        if (found != 0x7fffffff) atomicMin(&ired[0], found);
        if (lp >= 0) atomicMax(&ired[1], lp);
        __syncthreads();
        const int fb = ired[0];
        if (ired[1] > last_pos) last_pos = ired[1];
        __syncthreads();
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
    __syncthreads();
    if (threadIdx.x == 0) {
        int a = 0;
        for (int s = 0; s < S; ++s) { H.off[s] = a; a += H.cnt[s]; }
        H.off[S] = a;
    }
    __syncthreads();
}

// Gather every slice key that `keep(key)` accepts into list[0..*lcnt)
// (order arbitrary); keys beyond `cap` set *oflow.  All loads independent.
template <class F>
__device__ inline void gather_keys(const Workspace& W, int b, int S, const SliceHdrs& H, F keep,
                                   uint64_t* list, int cap, int* lcnt, int* oflow) {
    if (threadIdx.x == 0) { *lcnt = 0; *oflow = 0; }
    __syncthreads();
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
    __syncthreads();
}

}  // namespace spec
