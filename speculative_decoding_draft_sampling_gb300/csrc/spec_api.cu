// spec_api.cu -- the C ABI of libspecverify: argument checks, workspace
// layout, launch configuration.  Every device step runs in the kernels of
// this library; the host code only validates, lays out scratch space and
// enqueues work on the caller's stream (one 128-byte memset of the queue
// counters and one cluster launch per call).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/spec_verify.h"
#include "spec_chain.cuh"

namespace {

thread_local std::string g_err;

spec_status fail(spec_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

spec_status cuda_fail(cudaError_t e, const char* where) {
    return fail(SPEC_CUDA_ERROR, "%s: %s", where, cudaGetErrorString(e));
}

int g_tune_c = 0;        // CTAs per cluster (0 = automatic)
int g_tune_spc = 0;      // slots per CTA (0 = automatic)

constexpr int kDefaultC = 8;
constexpr int kDefaultSpc = 1;
constexpr int kMinSliceElems = 2048;   // a slice holds at least this many elements (small rows use small clusters)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_dtype(spec_dtype d) { return d == SPEC_F32 || d == SPEC_BF16; }
int esize_of(spec_dtype d) { return d == SPEC_F32 ? 4 : 2; }

// Where an array lives.  Device (and managed) memory is used as it is;
// pinned host memory is read and written in place through its mapping into
// the device's address space (on a Grace host, over the NVLink-C2C link);
// pageable host memory cannot be reached by the kernels and is refused.
template <class T>
spec_status map_ptr(const char* who, const char* name, T*& p) {
    if (!p) return SPEC_OK;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return fail(SPEC_INVALID_ARG, "%s: %s is not memory the device can reach", who, name);
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return SPEC_OK;
    if (a.type == cudaMemoryTypeHost && a.devicePointer) {
        p = static_cast<T*>(a.devicePointer);
        return SPEC_OK;
    }
    return fail(SPEC_INVALID_ARG, "%s: %s is pageable host memory (pass device memory or pinned host memory)", who,
                name);
}
#define SPEC_MAP(x)                                              \
    do {                                                         \
        const spec_status map_s_ = map_ptr(who, #x, x);          \
        if (map_s_ != SPEC_OK) return map_s_;                    \
    } while (0)

// The workspace holds the kernels' queues, flags and partial results: it must
// be device memory.
spec_status ws_on_device(const char* who, const void* ws) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ws) != cudaSuccess || a.type != cudaMemoryTypeDevice) {
        cudaGetLastError();
        return fail(SPEC_INVALID_ARG, "%s: the workspace must be device memory", who);
    }
    return SPEC_OK;
}
#define SPEC_WS_DEVICE(w)                                        \
    do {                                                         \
        const spec_status ws_s_ = ws_on_device(who, w);          \
        if (ws_s_ != SPEC_OK) return ws_s_;                      \
    } while (0)

// Bulk copies (TMA) need device memory: host memory mapped into the device's
// address space is read with plain loads.
bool device_memory(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int smem_optin() {
    int d = 0, v = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) != cudaSuccess) return 0;
    return v;
}

// CTAs per cluster for rows of V elements: each slice at least
// kMinSliceElems long; a power of two up to kDefaultC, or the tuned size.
int cluster_size_for(int V) {
    int by_v = (V + kMinSliceElems - 1) / kMinSliceElems;
    if (by_v < 1) by_v = 1;
    if (g_tune_c > 0) return g_tune_c < by_v ? g_tune_c : by_v;
    int c = 1;
    while (c * 2 <= kDefaultC && c * 2 <= by_v) c *= 2;
    return c;
}

// Launch plan of one call.
struct Plan {
    spec::EngArgs E;
    size_t smem;
    int clusters;   // clusters launched
    int resident;   // clusters the device holds at once
};

// Cached occupancy per (kernel, cluster size, shared memory) and device.
struct OccKey {
    const void* fn;
    int C;
    size_t smem;
    int dev;
    int n;
};
std::mutex g_occ_mu;
OccKey g_occ[64];
int g_occ_n = 0;

int max_clusters(const void* fn, int C, size_t smem, cudaError_t& err) {
    int dev = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return 0;
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        for (int i = 0; i < g_occ_n; ++i)
            if (g_occ[i].fn == fn && g_occ[i].C == C && g_occ[i].smem == smem && g_occ[i].dev == dev) return g_occ[i].n;
    }
    // every launch of this kernel may use up to the device's opt-in maximum
    // (set once, before the first query, whatever this call's size)
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin());
    if (err != cudaSuccess) return 0;
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    cfg.blockDim = dim3(spec::kBlockThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(C);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    err = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    if (err != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    if (g_occ_n < 64) g_occ[g_occ_n++] = OccKey{fn, C, smem, dev, n};
    return n;
}

// Geometry: cluster size, slots, slice length, ring depth (as many stages as
// fit next to the rest of the shared memory, at most kStages).  Requests
// spread over every cluster that fits on the device: a cluster keeps
// R = ceil(B / clusters) of them in flight (at most slots_per_cta per CTA),
// so small batches still use every SM.
template <class SmemFn>
spec_status make_plan_c(const char* who, const void* fn, int C, int V, int part_bytes, int B, SmemFn smem_of,
                        Plan& pl);

// The automatic cluster size also weighs how many SMs its clusters cover:
// clusters must fit inside a GPC, so the largest size can leave SMs idle.
// A smaller size of at least 4 CTAs is taken when it covers more SMs; 2-CTA
// clusters only when, besides, the batch holds at least two requests per
// cluster (rows then queue, and throughput, not the latency of one row,
// sets the time).
template <class SmemFn>
spec_status make_plan(const char* who, const void* fn, int V, int part_bytes, int B, SmemFn smem_of, Plan& pl) {
    const int C = cluster_size_for(V);
    spec_status s = make_plan_c(who, fn, C, V, part_bytes, B, smem_of, pl);
    if (s != SPEC_OK || g_tune_c > 0) return s;
    int cur = C;
    for (int c = C / 2; c >= 2; c /= 2) {
        Plan p;
        if (make_plan_c(who, fn, c, V, part_bytes, B, smem_of, p) != SPEC_OK) break;
        const long long cov = static_cast<long long>(p.resident) * c;
        const long long cov_cur = static_cast<long long>(pl.resident) * cur;
        if (cov * 20 > cov_cur * 21 && (c >= 4 || B >= 2 * p.resident)) {
            pl = p;
            cur = c;
        }
    }
    return SPEC_OK;
}

template <class SmemFn>
spec_status make_plan_c(const char* who, const void* fn, int C, int V, int part_bytes, int B, SmemFn smem_of,
                        Plan& pl) {
    int spc_max = g_tune_spc > 0 ? g_tune_spc : kDefaultSpc;
    if (spc_max > spec::kMaxOwn) spc_max = spec::kMaxOwn;
    if (C * spc_max > spec::kMaxSlots) spc_max = spec::kMaxSlots / C;
    const int optin = smem_optin();
    // large stages when at least two fit (fewer waits and releases per
    // byte), else small ones
    int chunk = spec::kChunkLarge;
    auto fit = [&](int own, int& stages, size_t& smem) {
        const size_t base = smem_of(C, own, part_bytes, 0, spec::kChunkSmall);
        stages = 0;
        if (optin <= 0 || base > static_cast<size_t>(optin)) return false;
        const size_t room = static_cast<size_t>(optin) - base;
        if (room >= 2ull * spec::kChunkLarge) {
            chunk = spec::kChunkLarge;
        } else if (room >= 2ull * spec::kChunkSmall) {
            chunk = spec::kChunkSmall;
        } else {
            return false;
        }
        stages = static_cast<int>(room / chunk);
        if (stages > spec::kStages) stages = spec::kStages;
        smem = smem_of(C, own, part_bytes, stages, chunk);
        return true;
    };
    int stages = 0;
    size_t smem = 0;
    while (spc_max > 1 && !fit(spc_max, stages, smem)) --spc_max;
    if (!fit(spc_max, stages, smem))
        return fail(SPEC_UNSUPPORTED, "%s: the kernel's shared memory does not fit this device", who);
    cudaError_t e;
    int n = max_clusters(fn, C, smem, e);
    if (e != cudaSuccess) return cuda_fail(e, who);
    if (n < 1) return fail(SPEC_CUDA_ERROR, "%s: no cluster of %d CTAs fits this device", who, C);
    int R = (B + n - 1) / n;
    if (R > C * spc_max) R = C * spc_max;
    if (R < 1) R = 1;
    const int own = (R + C - 1) / C;
    if (own < spc_max) {
        // fewer slots per CTA: less shared memory for partials, maybe more stages
        fit(own, stages, smem);
        const int n2 = max_clusters(fn, C, smem, e);
        if (e != cudaSuccess) return cuda_fail(e, who);
        if (n2 >= 1) n = n2;
    }
    pl.E.stages = stages;
    pl.E.chunk = chunk;
    pl.E.C = C;
    pl.E.R = R;
    pl.E.own = own;
    pl.E.SL = static_cast<int>(align_up(static_cast<size_t>((V + C - 1) / C), 64));
    pl.E.part_bytes = part_bytes;
    pl.smem = smem;
    const int need = (B + R - 1) / R;
    pl.clusters = n < need ? n : need;
    if (pl.clusters < 1) pl.clusters = 1;
    pl.resident = n;
    return SPEC_OK;
}

template <class Args>
spec_status launch(const char* who, const void* fn, const Plan& pl, Args& A, void* ws, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(ws, 0, 128, st);   // request counter and error word
    if (e != cudaSuccess) return cuda_fail(e, who);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.clusters * pl.E.C));
    cfg.blockDim = dim3(spec::kBlockThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(pl.E.C);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    void* args[] = {&A};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return cuda_fail(e, who);
    return SPEC_OK;
}

// workspace: the control block, then per-request scratch (tree build only)
constexpr size_t kCtrlBytes = sizeof(spec::Ctrl);
size_t ws_bytes_for(int B, size_t extra_per_req) {
    return kCtrlBytes + static_cast<size_t>(B) * align_up(extra_per_req, 256);
}
spec::Workspace make_ws(void* ws, size_t extra_per_req) {
    spec::Workspace W;
    W.ctrl = static_cast<spec::Ctrl*>(ws);
    W.extra = static_cast<unsigned char*>(ws) + kCtrlBytes;
    W.extra_stride = align_up(extra_per_req, 256);
    return W;
}

int chain_cap(int top_k) {
    if (top_k <= 0) return 0;
    int c = 2 * top_k;
    if (c < top_k + 64) c = top_k + 64;
    return c < 512 ? c : 512;
}

}  // namespace

namespace spec {
// lets other translation units of the library report an argument error
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace spec

extern "C" {

const char* spec_last_error(void) { return g_err.c_str(); }
int spec_version(void) { return 200; }

spec_status spec_set_tuning(int slices_per_row, int slots_per_cta) {
    if (slices_per_row < 0 || slices_per_row > spec::kMaxC || slots_per_cta < 0 || slots_per_cta > spec::kMaxOwn)
        return fail(SPEC_INVALID_ARG, "spec_set_tuning: slices_per_row in [0, %d], slots_per_cta in [0, %d]",
                    spec::kMaxC, spec::kMaxOwn);
    g_tune_c = slices_per_row;
    g_tune_spc = slots_per_cta;
    return SPEC_OK;
}

spec_status spec_workspace_error(const void* ws, void* stream, uint32_t* err_out) {
    if (!ws || !err_out) return fail(SPEC_INVALID_ARG, "spec_workspace_error: null pointer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, &static_cast<const spec::Ctrl*>(ws)->error, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_workspace_error");
    *err_out = v;
    return SPEC_OK;
}

// ---------------------------------------------------------------------------
// chain
// ---------------------------------------------------------------------------
size_t spec_verify_chain_workspace_size(int B, int K, int V, int top_k) {
    (void)top_k;
    if (B < 0 || K < 0 || V < 1) return 0;
    return ws_bytes_for(B, 0);
}

spec_status spec_verify_chain(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const float* q, int64_t q_batch_stride, int64_t q_row_stride,
    const int32_t* draft, const float* uniforms,
    int B, int K, int V, float temperature, int top_k,
    const int32_t* k_per_req, const int32_t* l_row_off, const int32_t* q_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status, float* diag,
    void* ws, size_t ws_bytes, void* stream) {
    const char* who = "spec_verify_chain";
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_INVALID_ARG, "%s: need B >= 0, K >= 0, V >= 1", who);
    if (K > 4096) return fail(SPEC_UNSUPPORTED, "%s: K > 4096", who);
    if (!valid_dtype(ldt)) return fail(SPEC_INVALID_ARG, "%s: unknown logits dtype %d", who, (int)ldt);
    if (!(temperature > 0.0f) || !(temperature < 3.0e38f))
        return fail(SPEC_INVALID_ARG, "%s: temperature must be finite and > 0", who);
    const bool ragged = k_per_req != nullptr;
    if ((l_row_off != nullptr) != (q_row_off != nullptr) || (!ragged && l_row_off != nullptr))
        return fail(SPEC_INVALID_ARG, "%s: l_row_off and q_row_off come together, and only with k_per_req", who);
    const bool packed = ragged && l_row_off != nullptr;
    if (B == 0) return SPEC_OK;
    if (!logits || !uniforms || !out_tokens || !num_accepted || !status || !ws || (K > 0 && (!q || !draft)))
        return fail(SPEC_INVALID_ARG, "%s: null pointer argument", who);
    if (l_row_stride < V || (K > 0 && q_row_stride < V) || l_batch_stride < 0 || q_batch_stride < 0)
        return fail(SPEC_INVALID_ARG, "%s: row strides must be >= V, batch strides >= 0", who);
    if (ws_bytes < ws_bytes_for(B, 0))
        return fail(SPEC_INVALID_ARG, "%s: workspace too small (%zu < %zu)", who, ws_bytes, ws_bytes_for(B, 0));
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "%s: workspace must be 16-byte aligned", who);
    SPEC_MAP(logits);
    SPEC_MAP(q);
    SPEC_MAP(draft);
    SPEC_MAP(uniforms);
    SPEC_MAP(k_per_req);
    SPEC_MAP(l_row_off);
    SPEC_MAP(q_row_off);
    SPEC_MAP(out_tokens);
    SPEC_MAP(num_accepted);
    SPEC_MAP(status);
    SPEC_MAP(diag);
    SPEC_WS_DEVICE(ws);
    const int es = esize_of(ldt);
    const bool topk = top_k > 0 && top_k < V;
    spec::ChainArgs A{};
    A.logits = logits; A.l_bs = l_batch_stride; A.l_rs = l_row_stride;
    A.q = q; A.q_bs = q_batch_stride; A.q_rs = q_row_stride;
    A.draft = draft; A.uniforms = uniforms;
    A.B = B; A.K = K; A.V = V; A.ldt = (int)ldt;
    A.Td = static_cast<double>(temperature);
    A.c2 = static_cast<float>(1.4426950408889634 / A.Td);
    A.top_k = topk ? top_k : 0;
    A.k_per_req = k_per_req; A.l_row_off = l_row_off; A.q_row_off = q_row_off;
    A.out_tokens = out_tokens; A.num_accepted = num_accepted; A.status = status; A.diag = diag;
    A.cap_p = chain_cap(A.top_k);
    A.tma_l = aligned16(logits) && (l_row_stride * es) % 16 == 0 && (packed || (l_batch_stride * es) % 16 == 0) &&
              device_memory(logits);
    A.tma_q = q && aligned16(q) && (q_row_stride * 4) % 16 == 0 && (packed || (q_batch_stride * 4) % 16 == 0) &&
              device_memory(q);
    const void* fn = spec::chain_kernel_ptr((int)ldt, topk);
    Plan pl;
    spec_status s = make_plan(who, fn, V, spec::chain_part_bytes(A.top_k, A.cap_p), B,
                              [](int C, int own, int pb, int stages, int chunk) { return spec::chain_smem(C, own, pb, stages, chunk); },
                              pl);
    if (s != SPEC_OK) return s;
    A.E = pl.E;
    A.E.W = make_ws(ws, 0);
    return launch(who, fn, pl, A, ws, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// greedy
// ---------------------------------------------------------------------------
size_t spec_verify_greedy_workspace_size(int B, int K, int V) {
    if (B < 0 || K < 0 || V < 1) return 0;
    return ws_bytes_for(B, 0);
}

spec_status spec_verify_greedy(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* draft, int B, int K, int V,
    const int32_t* k_per_req, const int32_t* l_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    void* ws, size_t ws_bytes, void* stream) {
    const char* who = "spec_verify_greedy";
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_INVALID_ARG, "%s: need B >= 0, K >= 0, V >= 1", who);
    if (K > 4096) return fail(SPEC_UNSUPPORTED, "%s: K > 4096", who);
    if (!valid_dtype(ldt)) return fail(SPEC_INVALID_ARG, "%s: unknown logits dtype", who);
    if (l_row_off != nullptr && k_per_req == nullptr)
        return fail(SPEC_INVALID_ARG, "%s: l_row_off needs k_per_req", who);
    const bool packed = l_row_off != nullptr;
    if (B == 0) return SPEC_OK;
    if (!logits || !out_tokens || !num_accepted || !status || !ws || (K > 0 && !draft))
        return fail(SPEC_INVALID_ARG, "%s: null pointer argument", who);
    if (l_row_stride < V || l_batch_stride < 0) return fail(SPEC_INVALID_ARG, "%s: row stride must be >= V", who);
    if (ws_bytes < ws_bytes_for(B, 0))
        return fail(SPEC_INVALID_ARG, "%s: workspace too small (%zu < %zu)", who, ws_bytes, ws_bytes_for(B, 0));
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "%s: workspace must be 16-byte aligned", who);
    SPEC_MAP(logits);
    SPEC_MAP(draft);
    SPEC_MAP(k_per_req);
    SPEC_MAP(l_row_off);
    SPEC_MAP(out_tokens);
    SPEC_MAP(num_accepted);
    SPEC_MAP(status);
    SPEC_WS_DEVICE(ws);
    const int es = esize_of(ldt);
    spec::WalkArgs A{};
    A.logits = logits; A.l_bs = l_batch_stride; A.l_rs = l_row_stride;
    A.B = B; A.K = K; A.V = V; A.ldt = (int)ldt;
    A.draft = draft; A.k_per_req = k_per_req; A.l_row_off = l_row_off;
    A.out_tokens = out_tokens; A.num_accepted = num_accepted; A.status = status;
    A.tma_l = aligned16(logits) && (l_row_stride * es) % 16 == 0 && (packed || (l_batch_stride * es) % 16 == 0) &&
              device_memory(logits);
    const void* fn = spec::walk_kernel_ptr((int)ldt, 0);
    Plan pl;
    spec_status s = make_plan(who, fn, V, spec::walk_part_bytes(), B,
                              [](int C, int own, int pb, int stages, int chunk) { return spec::walk_smem(C, own, pb, stages, chunk); },
                              pl);
    if (s != SPEC_OK) return s;
    A.E = pl.E;
    A.E.W = make_ws(ws, 0);
    return launch(who, fn, pl, A, ws, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// tree build
// ---------------------------------------------------------------------------
size_t spec_tree_build_workspace_size(int B, int L, int V, int budget) {
    if (B < 0 || L < 0 || L > 16 || V < 1 || budget < 1 || budget > 256) return 0;
    return ws_bytes_for(B, spec::build_extra_bytes(budget, L));
}

spec_status spec_tree_build(
    const float* q, int64_t q_batch_stride, int64_t q_row_stride,
    int B, int L, int V, int budget,
    int32_t* token, int32_t* parent, int32_t* depth, double* score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status,
    void* ws, size_t ws_bytes, void* stream) {
    const char* who = "spec_tree_build";
    if (B < 0 || L < 0 || V < 1 || budget < 1)
        return fail(SPEC_INVALID_ARG, "%s: need B >= 0, L >= 0, V >= 1, budget >= 1", who);
    if (L > 16 || budget > 256) return fail(SPEC_UNSUPPORTED, "%s: L <= 16 and budget <= 256", who);
    if (B == 0) return SPEC_OK;
    if (!token || !parent || !depth || !score || !anc_mask || !num_nodes || !status || !ws || (L > 0 && !q))
        return fail(SPEC_INVALID_ARG, "%s: null pointer argument", who);
    if (q_row_stride < V || q_batch_stride < 0) return fail(SPEC_INVALID_ARG, "%s: row stride must be >= V", who);
    const size_t need = ws_bytes_for(B, spec::build_extra_bytes(budget, L));
    if (ws_bytes < need) return fail(SPEC_INVALID_ARG, "%s: workspace too small (%zu < %zu)", who, ws_bytes, need);
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "%s: workspace must be 16-byte aligned", who);
    SPEC_MAP(q);
    SPEC_MAP(token);
    SPEC_MAP(parent);
    SPEC_MAP(depth);
    SPEC_MAP(score);
    SPEC_MAP(anc_mask);
    SPEC_MAP(num_nodes);
    SPEC_MAP(status);
    SPEC_WS_DEVICE(ws);
    spec::BuildArgs A{};
    A.q = q; A.q_bs = q_batch_stride; A.q_rs = q_row_stride;
    A.B = B; A.L = L; A.V = V; A.N = budget; A.M = budget - 1;
    A.token = token; A.parent = parent; A.depth = depth; A.score = score;
    A.anc_mask = reinterpret_cast<unsigned long long*>(anc_mask);
    A.num_nodes = num_nodes; A.status = status;
    A.cap_p = budget > 1 ? budget - 1 : 1;
    A.tma_q = q && aligned16(q) && (q_row_stride * 4) % 16 == 0 && (q_batch_stride * 4) % 16 == 0 && device_memory(q);
    const void* fn = spec::build_kernel_ptr();
    Plan pl;
    spec_status s = make_plan(who, fn, V, spec::build_part_bytes(A.M), B,
                              [&](int C, int own, int pb, int stages, int chunk) {
                                  return spec::build_smem(C, own, pb, stages, chunk, budget, L);
                              },
                              pl);
    if (s != SPEC_OK) return s;
    A.E = pl.E;
    A.E.W = make_ws(ws, spec::build_extra_bytes(budget, L));
    return launch(who, fn, pl, A, ws, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// EAGLE-2 dynamic tree
// ---------------------------------------------------------------------------
size_t spec_eagle_expand_workspace_size(int B, int F, int K2) {
    if (B < 0 || F < 1 || K2 < 1) return 0;
    return ws_bytes_for(B * F, spec::eagle_row_extra_bytes(K2));
}

spec_status spec_eagle_expand(
    const float* q, int64_t q_batch_stride, int64_t q_row_stride,
    int B, int F, int V, int K2, int Fn, int G,
    int32_t* token, int32_t* parent, int32_t* depth, double* score, int32_t* num_gen,
    const int32_t* front_in, const int32_t* num_front_in,
    int32_t* front_out, int32_t* num_front_out, int32_t* status,
    void* ws, size_t ws_bytes, void* stream) {
    const char* who = "spec_eagle_expand";
    if (B < 0 || F < 1 || V < 1 || K2 < 1 || Fn < 0 || G < 1)
        return fail(SPEC_INVALID_ARG, "%s: need B >= 0, F >= 1, V >= 1, K2 >= 1, Fn >= 0, G >= 1", who);
    if (F > 64 || K2 > 255 || Fn > 64 || F * K2 > 2048 || G > 8192)
        return fail(SPEC_UNSUPPORTED, "%s: F <= 64, K2 <= 255, Fn <= 64, F * K2 <= 2048, G <= 8192", who);
    if (B == 0) return SPEC_OK;
    if (!q || !token || !parent || !depth || !score || !num_gen || !front_in || !num_front_in ||
        (Fn > 0 && !front_out) || !num_front_out || !status || !ws)
        return fail(SPEC_INVALID_ARG, "%s: null pointer argument", who);
    if (q_row_stride < V || q_batch_stride < 0) return fail(SPEC_INVALID_ARG, "%s: row stride must be >= V", who);
    const size_t need = ws_bytes_for(B * F, spec::eagle_row_extra_bytes(K2));
    if (ws_bytes < need) return fail(SPEC_INVALID_ARG, "%s: workspace too small (%zu < %zu)", who, ws_bytes, need);
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "%s: workspace must be 16-byte aligned", who);
    SPEC_MAP(q);
    SPEC_MAP(token);
    SPEC_MAP(parent);
    SPEC_MAP(depth);
    SPEC_MAP(score);
    SPEC_MAP(num_gen);
    SPEC_MAP(front_in);
    SPEC_MAP(num_front_in);
    SPEC_MAP(front_out);
    SPEC_MAP(num_front_out);
    SPEC_MAP(status);
    SPEC_WS_DEVICE(ws);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    spec::EagleArgs A{};
    A.base.q = q; A.base.q_bs = q_batch_stride; A.base.q_rs = q_row_stride;
    A.base.B = B; A.base.L = 1; A.base.V = V; A.base.N = K2 + 1; A.base.M = K2;
    A.base.cap_p = K2;
    A.base.tma_q = aligned16(q) && (q_row_stride * 4) % 16 == 0 && (q_batch_stride * 4) % 16 == 0 && device_memory(q);
    A.F = F; A.G = G; A.front_in = front_in; A.num_front_in = num_front_in; A.num_gen = num_gen;
    A.score = score; A.depth = depth;
    const void* fn = spec::eagle_rows_kernel_ptr();
    Plan pl;
    spec_status s = make_plan(who, fn, V, spec::build_part_bytes(K2), B * F,
                              [](int C, int own, int pb, int stages, int chunk) {
                                  return spec::eagle_rows_smem(C, own, pb, stages, chunk);
                              },
                              pl);
    if (s != SPEC_OK) return s;
    A.base.E = pl.E;
    A.base.E.W = make_ws(ws, spec::eagle_row_extra_bytes(K2));
    s = launch(who, fn, pl, A, ws, st);
    if (s != SPEC_OK) return s;
    spec::EagleGrowArgs g{};
    g.rows = static_cast<const unsigned char*>(ws) + kCtrlBytes;
    g.row_stride = static_cast<long long>(align_up(spec::eagle_row_extra_bytes(K2), 256));
    g.B = B; g.F = F; g.K2 = K2; g.Fn = Fn; g.G = G;
    g.token = token; g.parent = parent; g.depth = depth; g.score = score; g.num_gen = num_gen;
    g.front_in = front_in; g.num_front_in = num_front_in;
    g.front_out = front_out; g.num_front_out = num_front_out; g.status = status;
    const cudaError_t e = spec::eagle_grow_run(g, st);
    if (e != cudaSuccess) return cuda_fail(e, who);
    return SPEC_OK;
}

spec_status spec_eagle_rerank(
    const int32_t* token, const int32_t* parent, const int32_t* depth, const double* score,
    const int32_t* num_gen, int B, int G, int budget,
    int32_t* out_token, int32_t* out_parent, int32_t* out_depth, double* out_score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status, void* stream) {
    const char* who = "spec_eagle_rerank";
    if (B < 0 || G < 1 || budget < 1) return fail(SPEC_INVALID_ARG, "%s: need B >= 0, G >= 1, budget >= 1", who);
    if (G > 8192 || budget > 1024) return fail(SPEC_UNSUPPORTED, "%s: G <= 8192 and budget <= 1024", who);
    if (B == 0) return SPEC_OK;
    if (!token || !parent || !depth || !score || !num_gen || !out_token || !out_parent || !out_depth || !out_score ||
        !anc_mask || !num_nodes || !status)
        return fail(SPEC_INVALID_ARG, "%s: null pointer argument", who);
    SPEC_MAP(token);
    SPEC_MAP(parent);
    SPEC_MAP(depth);
    SPEC_MAP(score);
    SPEC_MAP(num_gen);
    SPEC_MAP(out_token);
    SPEC_MAP(out_parent);
    SPEC_MAP(out_depth);
    SPEC_MAP(out_score);
    SPEC_MAP(anc_mask);
    SPEC_MAP(num_nodes);
    SPEC_MAP(status);
    spec::EagleRerankArgs A{};
    A.token = token; A.parent = parent; A.depth = depth; A.score = score; A.num_gen = num_gen;
    A.B = B; A.G = G; A.N = budget;
    A.out_token = out_token; A.out_parent = out_parent; A.out_depth = out_depth; A.out_score = out_score;
    A.anc_mask = reinterpret_cast<unsigned long long*>(anc_mask); A.num_nodes = num_nodes; A.status = status;
    const cudaError_t e = spec::eagle_rerank_run(A, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return SPEC_OK;
}

// ---------------------------------------------------------------------------
// tree walk
// ---------------------------------------------------------------------------
size_t spec_verify_tree_workspace_size(int B, int N, int V) {
    if (B < 0 || N < 1 || V < 1) return 0;
    return ws_bytes_for(B, 0);
}

spec_status spec_verify_tree(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes,
    int B, int N, int V, int max_depth,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    void* ws, size_t ws_bytes, void* stream) {
    const char* who = "spec_verify_tree";
    if (B < 0 || N < 1 || V < 1 || max_depth < 0)
        return fail(SPEC_INVALID_ARG, "%s: need B >= 0, N >= 1, V >= 1, max_depth >= 0", who);
    if (!valid_dtype(ldt)) return fail(SPEC_INVALID_ARG, "%s: unknown logits dtype", who);
    if (N > 8192) return fail(SPEC_UNSUPPORTED, "%s: N > 8192", who);
    if (B == 0) return SPEC_OK;
    if (!logits || !token || !parent || !num_nodes || !path_nodes || !out_tokens || !num_accepted || !status || !ws)
        return fail(SPEC_INVALID_ARG, "%s: null pointer argument", who);
    if (l_row_stride < V || l_batch_stride < 0) return fail(SPEC_INVALID_ARG, "%s: row stride must be >= V", who);
    if (ws_bytes < ws_bytes_for(B, 0))
        return fail(SPEC_INVALID_ARG, "%s: workspace too small (%zu < %zu)", who, ws_bytes, ws_bytes_for(B, 0));
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "%s: workspace must be 16-byte aligned", who);
    SPEC_MAP(logits);
    SPEC_MAP(token);
    SPEC_MAP(parent);
    SPEC_MAP(num_nodes);
    SPEC_MAP(path_nodes);
    SPEC_MAP(out_tokens);
    SPEC_MAP(num_accepted);
    SPEC_MAP(status);
    SPEC_WS_DEVICE(ws);
    const int es = esize_of(ldt);
    spec::WalkArgs A{};
    A.logits = logits; A.l_bs = l_batch_stride; A.l_rs = l_row_stride;
    A.B = B; A.K = 0; A.V = V; A.ldt = (int)ldt;
    A.token = token; A.parent = parent; A.num_nodes = num_nodes; A.N = N; A.L = max_depth;
    A.path_nodes = path_nodes; A.out_tokens = out_tokens; A.num_accepted = num_accepted; A.status = status;
    A.tma_l = aligned16(logits) && (l_row_stride * es) % 16 == 0 && (l_batch_stride * es) % 16 == 0 &&
              device_memory(logits);
    const void* fn = spec::walk_kernel_ptr((int)ldt, 1);
    Plan pl;
    spec_status s = make_plan(who, fn, V, spec::walk_part_bytes(), B,
                              [](int C, int own, int pb, int stages, int chunk) { return spec::walk_smem(C, own, pb, stages, chunk); },
                              pl);
    if (s != SPEC_OK) return s;
    A.E = pl.E;
    A.E.W = make_ws(ws, 0);
    return launch(who, fn, pl, A, ws, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// stochastic tree walk
// ---------------------------------------------------------------------------
size_t spec_verify_tree_sample_workspace_size(int B, int N, int V) {
    if (B < 0 || N < 1 || V < 1) return 0;
    return ws_bytes_for(B, 0);
}

spec_status spec_verify_tree_sample(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes, const float* uniforms,
    int B, int N, int V, int max_depth, float temperature, int top_k,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    void* ws, size_t ws_bytes, void* stream) {
    const char* who = "spec_verify_tree_sample";
    if (B < 0 || N < 1 || V < 1 || max_depth < 0)
        return fail(SPEC_INVALID_ARG, "%s: need B >= 0, N >= 1, V >= 1, max_depth >= 0", who);
    if (!valid_dtype(ldt)) return fail(SPEC_INVALID_ARG, "%s: unknown logits dtype", who);
    if (!(temperature > 0.0f) || !(temperature < 3.0e38f))
        return fail(SPEC_INVALID_ARG, "%s: temperature must be finite and > 0", who);
    if (N > 8192 || max_depth > 4096) return fail(SPEC_UNSUPPORTED, "%s: N > 8192 or max_depth > 4096", who);
    if (B == 0) return SPEC_OK;
    if (!logits || !token || !parent || !num_nodes || !uniforms || !path_nodes || !out_tokens || !num_accepted ||
        !status || !ws)
        return fail(SPEC_INVALID_ARG, "%s: null pointer argument", who);
    if (l_row_stride < V || l_batch_stride < 0) return fail(SPEC_INVALID_ARG, "%s: row stride must be >= V", who);
    if (ws_bytes < ws_bytes_for(B, 0))
        return fail(SPEC_INVALID_ARG, "%s: workspace too small (%zu < %zu)", who, ws_bytes, ws_bytes_for(B, 0));
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "%s: workspace must be 16-byte aligned", who);
    SPEC_MAP(logits);
    SPEC_MAP(token);
    SPEC_MAP(parent);
    SPEC_MAP(num_nodes);
    SPEC_MAP(uniforms);
    SPEC_MAP(path_nodes);
    SPEC_MAP(out_tokens);
    SPEC_MAP(num_accepted);
    SPEC_MAP(status);
    SPEC_WS_DEVICE(ws);
    const int es = esize_of(ldt);
    const bool topk = top_k > 0 && top_k < V;
    spec::ChainArgs A{};
    A.logits = logits; A.l_bs = l_batch_stride; A.l_rs = l_row_stride;
    A.uniforms = uniforms;
    A.B = B; A.K = 0; A.V = V; A.ldt = (int)ldt;
    A.Td = static_cast<double>(temperature);
    A.c2 = static_cast<float>(1.4426950408889634 / A.Td);
    A.top_k = topk ? top_k : 0;
    A.out_tokens = out_tokens; A.num_accepted = num_accepted; A.status = status;
    A.cap_p = chain_cap(A.top_k);
    A.tma_l = aligned16(logits) && (l_row_stride * es) % 16 == 0 && (l_batch_stride * es) % 16 == 0 &&
              device_memory(logits);
    A.tree = 1;
    A.t_token = token; A.t_parent = parent; A.t_nn = num_nodes; A.N = N; A.L = max_depth;
    A.path_nodes = path_nodes;
    const void* fn = spec::chain_kernel_ptr((int)ldt, topk);
    Plan pl;
    spec_status s = make_plan(who, fn, V, spec::chain_part_bytes(A.top_k, A.cap_p), B,
                              [](int C, int own, int pb, int stages, int chunk) { return spec::chain_smem(C, own, pb, stages, chunk); },
                              pl);
    if (s != SPEC_OK) return s;
    A.E = pl.E;
    A.E.W = make_ws(ws, 0);
    return launch(who, fn, pl, A, ws, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// accepted-path KV compaction
// ---------------------------------------------------------------------------
spec_status spec_kv_compact(
    const void* src, int64_t src_plane_stride, int64_t src_batch_stride, int64_t src_row_stride,
    void* dst, int64_t dst_plane_stride, int64_t dst_batch_stride, int64_t dst_row_stride,
    int P, int B, int N, int64_t row_bytes,
    const int32_t* path_nodes, int path_width, const int32_t* num_accepted, const int32_t* dst_pos,
    void* stream) {
    const char* who = "spec_kv_compact";
    if (P < 0 || B < 0 || N < 1 || path_width < 1 || row_bytes < 1)
        return fail(SPEC_INVALID_ARG, "%s: need P >= 0, B >= 0, N >= 1, path_width >= 1, row_bytes >= 1", who);
    if (P == 0 || B == 0) return SPEC_OK;
    if (!src || !dst || !path_nodes || !num_accepted) return fail(SPEC_INVALID_ARG, "%s: null pointer argument", who);
    if (src_row_stride < row_bytes || dst_row_stride < row_bytes || src_batch_stride < 0 || dst_batch_stride < 0 ||
        src_plane_stride < 0 || dst_plane_stride < 0)
        return fail(SPEC_INVALID_ARG, "%s: row strides must be >= row_bytes, other strides >= 0", who);
    SPEC_MAP(src);
    SPEC_MAP(dst);
    SPEC_MAP(path_nodes);
    SPEC_MAP(num_accepted);
    SPEC_MAP(dst_pos);
    spec::KvArgs A{};
    A.src = static_cast<const unsigned char*>(src);
    A.s_plane = src_plane_stride; A.s_batch = src_batch_stride; A.s_row = src_row_stride;
    A.dst = static_cast<unsigned char*>(dst);
    A.d_plane = dst_plane_stride; A.d_batch = dst_batch_stride; A.d_row = dst_row_stride;
    A.P = P; A.B = B; A.N = N; A.W = path_width; A.row_bytes = row_bytes;
    A.path_nodes = path_nodes; A.num_accepted = num_accepted; A.dst_pos = dst_pos;
    auto all_mult = [&](long long m) {
        const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
        return s0 % m == 0 && d0 % m == 0 && row_bytes % m == 0 && src_row_stride % m == 0 &&
               dst_row_stride % m == 0 && src_batch_stride % m == 0 && dst_batch_stride % m == 0 &&
               src_plane_stride % m == 0 && dst_plane_stride % m == 0;
    };
    A.width = all_mult(16) ? 16 : (all_mult(4) ? 4 : 1);
    int d = 0, sms = 0;
    cudaGetDevice(&d);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    cudaError_t e = spec::kv_compact_run(A, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, who);
    return SPEC_OK;
}

// ---------------------------------------------------------------------------
// adaptive length
// ---------------------------------------------------------------------------
spec_status spec_adaptive_len(
    const float* conf, int B, int Kmax, float a, float b,
    int32_t* k_out, double* surv, double* exp_adv,
    int32_t* l_row_off, int32_t* q_row_off, void* stream) {
    if (B < 0 || Kmax < 0) return fail(SPEC_INVALID_ARG, "spec_adaptive_len: need B >= 0, Kmax >= 0");
    if (!(a > 0.0f) || !(b >= 0.0f) || !(a < 3.0e38f) || !(b < 3.0e38f))
        return fail(SPEC_INVALID_ARG, "spec_adaptive_len: need finite a > 0 and b >= 0");
    if (!k_out || !l_row_off || !q_row_off || (B > 0 && Kmax > 0 && !conf))
        return fail(SPEC_INVALID_ARG, "spec_adaptive_len: null pointer argument");
    if (static_cast<long long>(B) * (Kmax + 1) > 0x7fffffffLL)
        return fail(SPEC_UNSUPPORTED, "spec_adaptive_len: row offsets overflow int32");
    const char* who = "spec_adaptive_len";
    SPEC_MAP(conf);
    SPEC_MAP(k_out);
    SPEC_MAP(surv);
    SPEC_MAP(exp_adv);
    SPEC_MAP(l_row_off);
    SPEC_MAP(q_row_off);
    cudaError_t e = spec::adaptive_run(conf, B, Kmax, a, b, nullptr, k_out, surv, exp_adv, l_row_off, q_row_off,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "spec_adaptive_len: launch");
    return SPEC_OK;
}

spec_status spec_adaptive_len_table(
    const float* conf, int B, int Kmax, const double* cost,
    int32_t* k_out, double* surv, double* exp_adv,
    int32_t* l_row_off, int32_t* q_row_off, void* stream) {
    if (B < 0 || Kmax < 0) return fail(SPEC_INVALID_ARG, "spec_adaptive_len_table: need B >= 0, Kmax >= 0");
    if (!cost || !k_out || !l_row_off || !q_row_off || (B > 0 && Kmax > 0 && !conf))
        return fail(SPEC_INVALID_ARG, "spec_adaptive_len_table: null pointer argument");
    if (static_cast<long long>(B) * (Kmax + 1) > 0x7fffffffLL)
        return fail(SPEC_UNSUPPORTED, "spec_adaptive_len_table: row offsets overflow int32");
    const char* who = "spec_adaptive_len_table";
    SPEC_MAP(conf);
    SPEC_MAP(cost);
    SPEC_MAP(k_out);
    SPEC_MAP(surv);
    SPEC_MAP(exp_adv);
    SPEC_MAP(l_row_off);
    SPEC_MAP(q_row_off);
    cudaError_t e = spec::adaptive_run(conf, B, Kmax, 1.0f, 0.0f, cost, k_out, surv, exp_adv, l_row_off, q_row_off,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "spec_adaptive_len_table: launch");
    return SPEC_OK;
}

}  // extern "C"
