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

constexpr int kChunkBytes = 12288;   // one ring stage
constexpr int kStages = 4;           // ring depth: 48 KiB in flight per CTA
constexpr int kMaxSlices = 32;

enum : uint32_t { kErrWait = 1u, kErrQueue = 2u };

struct Ctrl {
    uint32_t head;     // next unit index to claim
    uint32_t tail;     // pushed tasks
    uint32_t done;     // finished requests
    uint32_t error;    // kErr* bits
    uint32_t pad[60];
};
static_assert(sizeof(Ctrl) == 256, "Ctrl is one 256-byte block");

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
    float vmax;        // slice maximum
    int32_t cnt;       // number of keys written
    uint32_t flags;    // kPf* bits
    int32_t pad0;
    uint64_t kth;      // slice-local threshold key (top-k) / best key (argmax)
    double sum;        // slice sum (meaning depends on the op)
    double sum2;
    uint64_t pad1[3];
};
static_assert(sizeof(PartHdr) == 64, "PartHdr is 64 bytes");
enum : uint32_t { kPfBad = 1u, kPfOverflow = 2u };

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
};

__device__ __forceinline__ PartHdr* part_hdr(const Workspace& W, int b, int s, int S) {
    return reinterpret_cast<PartHdr*>(W.part + (static_cast<size_t>(b) * S + s) * W.part_stride);
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
                    if (ns < 1024) ns <<= 1;
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
        __threadfence();
        const uint32_t prev = atomicAdd(&W.counter[b], 1u);
        int last = (prev == static_cast<uint32_t>(S - 1));
        if (last) {
            __threadfence();
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
    __threadfence();
    const uint32_t ti = atomicAdd(&W.ctrl->tail, 1u);
    if (ti >= W.maxt) { atomicOr(&W.ctrl->error, kErrQueue); return; }
    __stcg(&W.tasks[ti].b, t.b);
    __stcg(&W.tasks[ti].row, t.row);
    __stcg(&W.tasks[ti].kind, t.kind);
    __stcg(&W.tasks[ti].aux, t.aux);
    __threadfence();
    st_release(&W.ready[ti], 1u);
}

// Thread 0 of the combining CTA, after the request's outputs are written by
// the whole CTA (call after a __syncthreads()).
__device__ __forceinline__ void finish_request(const Workspace& W) {
    __threadfence();
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
// through the ring.  Calls, on every thread:
//   fn.pre_vec(active, vals, x) / fn.pre_end()   -- first chunk only, if Fn::kPrepass
//   fn.vec(active, vals, x)                      -- one 16-byte vector per thread
//   fn.round_end()                               -- after each round of vectors
// Tail elements that do not fill a 16-byte vector go through fn.vec with
// only vals[0] meaningful and `n` = 1 via fn.scalar(active, v, x).
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
        if (Fn::kPrepass && c == 0) {
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
        __syncthreads();   // every thread is done with stage s
        if (tma && threadIdx.x == 0 && c + kStages < nch) {
            const int c2 = c + kStages;
            const int ne2 = min(CE, n - c2 * CE);
            R.issue(s, base + static_cast<long long>(c2) * kChunkBytes, (ne2 * E::kBytes) & ~15);
        }
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
// smallest x with C(x) > t.  Blocks of kThreads*4 consecutive elements; each
// thread owns 4 consecutive elements (fp32 prefix inside, fp64 across).
// If rounding leaves no crossing, returns the last x with w(x) > 0 (or x0).
template <class W>
__device__ int cta_icdf(int x0, int x1, double t, W& w, double* red, int* ired) {
    double base = 0.0;
    int last_pos = -1;
    for (int b0 = x0; b0 < x1; b0 += kThreads * 4) {
        const int xs = b0 + threadIdx.x * 4;
        float wv[4];
        float loc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int x = xs + j;
            wv[j] = (x < x1) ? w(x) : 0.f;
            loc += wv[j];
        }
        int lp = -1;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (wv[j] > 0.f) lp = xs + j;
        double tot;
        const double ex = block_exscan_d(static_cast<double>(loc), red, tot);
        // crossing thread: base+ex <= t < base+ex+loc
        int found = 0x7fffffff;
        if (loc > 0.f && base + ex + static_cast<double>(loc) > t) {
            double c = base + ex;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                c += static_cast<double>(wv[j]);
                if (wv[j] > 0.f && c > t) { found = xs + j; break; }
            }
        }
        // lowest crossing index across the block; also the last positive x
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

}  // namespace spec
