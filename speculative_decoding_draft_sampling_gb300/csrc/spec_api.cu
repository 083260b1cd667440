// spec_api.cu -- the C ABI of libspecverify: argument checks, workspace
// layout, launch configuration.  Every device step runs in the kernels of
// this library; the host code only validates, lays out scratch space and
// enqueues work on the caller's stream (one memset of the queue counters and
// one kernel per call).
#include <cstdarg>
#include <cstdio>
#include <cstring>
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

int g_tune_slices = 0;
int g_tune_ctas = 0;

struct DevInfo {
    int sms = 0;
};
DevInfo g_dev[64];

int sm_count() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return 0;
    if (g_dev[d].sms == 0) cudaDeviceGetAttribute(&g_dev[d].sms, cudaDevAttrMultiProcessorCount, d);
    return g_dev[d].sms;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    size_t off_ready, off_counter, zero_bytes, off_req, off_part, off_extra, off_persist, total;
    uint32_t maxt, maxu, part_stride;
    uint64_t extra_stride;
    int smax;
};

// slices per row never exceed kMaxSlices nor ceil(V / 64) (slices are >= 64 elements)
int max_slices_for(int V) {
    const int s = (V + 63) / 64;
    return s < spec::kMaxSlices ? s : spec::kMaxSlices;
}

Layout make_layout(int B, long long maxt, int cap_p, size_t extra_per_req, int smax) {
    Layout L{};
    L.maxt = static_cast<uint32_t>(maxt);
    L.smax = smax;
    L.maxu = static_cast<uint32_t>(maxt * smax);   // a pushed task has at most smax slices
    L.off_ready = sizeof(spec::Ctrl);
    L.off_counter = align_up(L.off_ready + 16ull * L.maxu, 16);   // 16-byte unit records
    L.zero_bytes = align_up(L.off_counter + 4ull * B, 256);
    L.off_req = L.zero_bytes;
    L.off_part = align_up(L.off_req + sizeof(spec::ReqState) * B, 256);
    // room for the (up to 2 * kPreKeys) keys a combine fetches with the header
    const int keys = cap_p > 2 * spec::kPreKeys ? cap_p : 2 * spec::kPreKeys;
    L.part_stride = static_cast<uint32_t>(align_up(sizeof(spec::PartHdr) + 8ull * keys, 128));
    L.off_extra = align_up(L.off_part + static_cast<size_t>(B) * smax * L.part_stride, 256);
    L.extra_stride = align_up(extra_per_req, 256);
    L.off_persist = align_up(L.off_extra + static_cast<size_t>(B) * L.extra_stride, 128);
    L.total = L.off_persist + 128;
    return L;
}

spec::Workspace make_ws(void* ws, const Layout& L) {
    unsigned char* p = static_cast<unsigned char*>(ws);
    spec::Workspace W;
    W.ctrl = reinterpret_cast<spec::Ctrl*>(p);
    W.urec = reinterpret_cast<unsigned long long*>(p + L.off_ready);
    W.counter = reinterpret_cast<uint32_t*>(p + L.off_counter);
    W.req = reinterpret_cast<spec::ReqState*>(p + L.off_req);
    W.part = p + L.off_part;
    W.extra = p + L.off_extra;
    W.persist = reinterpret_cast<uint32_t*>(p + L.off_persist);
    W.part_stride = L.part_stride;
    W.maxt = L.maxt;
    W.maxu = L.maxu;
    W.extra_stride = L.extra_stride;
    W.smax = L.smax;
    return W;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#ifndef SPEC_FIRST_FACTOR
#define SPEC_FIRST_FACTOR 4   // first-row units per CTA
#endif
// Slices per row: enough units to give every CTA several at the start, each
// slice at least 32 KiB of row (a unit's fixed costs stay small next to its
// stream), at most `max_s`.
void choose_slices(int B, int V, int esize, int grid, int max_s, int& S, int& SL) {
    int s;
    if (g_tune_slices > 0) {
        s = g_tune_slices;
    } else {
        s = static_cast<int>((static_cast<long long>(SPEC_FIRST_FACTOR) * grid + B - 1) / (B > 0 ? B : 1));
        const long long row_bytes = static_cast<long long>(V) * esize;
        const int by_size = static_cast<int>((row_bytes + 32767) / 32768);
        if (s > by_size) s = by_size;
    }
    if (s > max_s) s = max_s;
    if (s > spec::kMaxSlices) s = spec::kMaxSlices;
    if (s < 1) s = 1;
    SL = static_cast<int>(align_up(static_cast<size_t>((V + s - 1) / s), 64));
    S = (V + SL - 1) / SL;
    if (S < 1) S = 1;
}

int grid_for(int occ, int units) {
    int per = occ;
    if (g_tune_ctas > 0 && g_tune_ctas < per) per = g_tune_ctas;
    if (per < 1) per = 1;
    long long g = static_cast<long long>(sm_count()) * per;
    if (g > units) g = units;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

int chain_cap_p(int B, int K, int V, int top_k) {
    (void)B; (void)K;
    if (top_k <= 0 || top_k >= V) return 0;
    int c = top_k * 2;
    if (c < top_k + 64) c = top_k + 64;
    return c;
}

bool valid_dtype(spec_dtype d) { return d == SPEC_F32 || d == SPEC_BF16; }
int esize_of(spec_dtype d) { return d == SPEC_F32 ? 4 : 2; }

}  // namespace

namespace spec {
// lets other translation units of the library report an argument error
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace spec

extern "C" {

const char* spec_last_error(void) { return g_err.c_str(); }
int spec_version(void) { return 100; }

spec_status spec_set_tuning(int slices_per_row, int ctas_per_sm) {
    if (slices_per_row < 0 || slices_per_row > spec::kMaxSlices || ctas_per_sm < 0)
        return fail(SPEC_INVALID_ARG, "spec_set_tuning: slices_per_row in [0, %d], ctas_per_sm >= 0",
                    spec::kMaxSlices);
    g_tune_slices = slices_per_row;
    g_tune_ctas = ctas_per_sm;
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
static Layout chain_layout(int B, int K, int V, int top_k) {
    // per request: every row at most twice (a hinted pass and its retry) plus a residual pass
    return make_layout(B, static_cast<long long>(B) * (2 * K + 4), chain_cap_p(B, K, V, top_k), 0, max_slices_for(V));
}

size_t spec_verify_chain_workspace_size(int B, int K, int V, int top_k) {
    if (B < 0 || K < 0 || V < 1) return 0;
    return chain_layout(B, K, V, top_k).total;
}

spec_status spec_verify_chain(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const float* q, int64_t q_batch_stride, int64_t q_row_stride,
    const int32_t* draft, const float* uniforms,
    int B, int K, int V, float temperature, int top_k,
    const int32_t* k_per_req, const int32_t* l_row_off, const int32_t* q_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status, float* diag,
    void* ws, size_t ws_bytes, void* stream) {
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_INVALID_ARG, "spec_verify_chain: need B >= 0, K >= 0, V >= 1");
    if (K > 4096) return fail(SPEC_UNSUPPORTED, "spec_verify_chain: K > 4096");
    if (B > spec::kMaxRecB) return fail(SPEC_UNSUPPORTED, "spec_verify_chain: B > %d", spec::kMaxRecB);
    if (!valid_dtype(ldt)) return fail(SPEC_INVALID_ARG, "spec_verify_chain: unknown logits dtype %d", (int)ldt);
    if (!(temperature > 0.0f) || !(temperature < 3.0e38f))
        return fail(SPEC_INVALID_ARG, "spec_verify_chain: temperature must be finite and > 0");
    const bool ragged = k_per_req != nullptr;
    if (ragged != (l_row_off != nullptr) || ragged != (q_row_off != nullptr))
        return fail(SPEC_INVALID_ARG, "spec_verify_chain: k_per_req, l_row_off, q_row_off: all or none");
    if (B == 0) return SPEC_OK;
    if (!logits || !uniforms || !out_tokens || !num_accepted || !status || !ws || (K > 0 && (!q || !draft)))
        return fail(SPEC_INVALID_ARG, "spec_verify_chain: null pointer argument");
    if (l_row_stride < V || (K > 0 && q_row_stride < V) || l_batch_stride < 0 || q_batch_stride < 0)
        return fail(SPEC_INVALID_ARG, "spec_verify_chain: row strides must be >= V, batch strides >= 0");
    const Layout Lw = chain_layout(B, K, V, top_k);
    if (ws_bytes < Lw.total)
        return fail(SPEC_INVALID_ARG, "spec_verify_chain: workspace too small (%zu < %zu)", ws_bytes, Lw.total);
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "spec_verify_chain: workspace must be 16-byte aligned");
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
    A.W = make_ws(ws, Lw);
    A.cap_p = chain_cap_p(B, K, V, top_k);
    A.tma_l = aligned16(logits) && (l_row_stride * es) % 16 == 0 && (ragged || (l_batch_stride * es) % 16 == 0);
    A.tma_q = q && aligned16(q) && (q_row_stride * 4) % 16 == 0 && (ragged || (q_batch_stride * 4) % 16 == 0);
    const int occ = spec::chain_occupancy((int)ldt, topk);
    if (occ < 1) return fail(SPEC_CUDA_ERROR, "spec_verify_chain: kernel does not fit on this device");
    int S, SL;
    // the combine gathers every slice's keys into 2048 slots
    const int max_s = topk ? (2048 / (A.cap_p > 0 ? A.cap_p : 1)) : spec::kMaxSlices;
    choose_slices(B, V, es, grid_for(occ, 1 << 30), max_s, S, SL);
    A.S = S; A.SL = SL;
    A.S1 = max_s < max_slices_for(V) ? max_s : max_slices_for(V);
    const int grid = grid_for(occ, B * S);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, Lw.zero_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_verify_chain: memset");
    e = spec::chain_run(A, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_verify_chain: launch");
    return SPEC_OK;
}

// ---------------------------------------------------------------------------
// greedy
// ---------------------------------------------------------------------------
static Layout greedy_layout(int B, int K, int V) {
    return make_layout(B, static_cast<long long>(B) * (K + 1), 0, 0, max_slices_for(V));
}

size_t spec_verify_greedy_workspace_size(int B, int K, int V) {
    if (B < 0 || K < 0 || V < 1) return 0;
    return greedy_layout(B, K, V).total;
}

spec_status spec_verify_greedy(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* draft, int B, int K, int V,
    const int32_t* k_per_req, const int32_t* l_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    void* ws, size_t ws_bytes, void* stream) {
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_INVALID_ARG, "spec_verify_greedy: need B >= 0, K >= 0, V >= 1");
    if (K > 4096) return fail(SPEC_UNSUPPORTED, "spec_verify_greedy: K > 4096");
    if (B > spec::kMaxRecB) return fail(SPEC_UNSUPPORTED, "spec_verify_greedy: B > %d", spec::kMaxRecB);
    if (!valid_dtype(ldt)) return fail(SPEC_INVALID_ARG, "spec_verify_greedy: unknown logits dtype");
    const bool ragged = k_per_req != nullptr;
    if (ragged != (l_row_off != nullptr))
        return fail(SPEC_INVALID_ARG, "spec_verify_greedy: k_per_req and l_row_off: both or neither");
    if (B == 0) return SPEC_OK;
    if (!logits || !out_tokens || !num_accepted || !status || !ws || (K > 0 && !draft))
        return fail(SPEC_INVALID_ARG, "spec_verify_greedy: null pointer argument");
    if (l_row_stride < V || l_batch_stride < 0)
        return fail(SPEC_INVALID_ARG, "spec_verify_greedy: row stride must be >= V");
    const Layout Lw = greedy_layout(B, K, V);
    if (ws_bytes < Lw.total)
        return fail(SPEC_INVALID_ARG, "spec_verify_greedy: workspace too small (%zu < %zu)", ws_bytes, Lw.total);
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "spec_verify_greedy: workspace must be 16-byte aligned");
    const int es = esize_of(ldt);
    spec::WalkArgs A{};
    A.logits = logits; A.l_bs = l_batch_stride; A.l_rs = l_row_stride;
    A.B = B; A.K = K; A.V = V; A.ldt = (int)ldt;
    A.draft = draft; A.k_per_req = k_per_req; A.l_row_off = l_row_off;
    A.out_tokens = out_tokens; A.num_accepted = num_accepted; A.status = status;
    A.W = make_ws(ws, Lw);
    A.tma_l = aligned16(logits) && (l_row_stride * es) % 16 == 0 && (ragged || (l_batch_stride * es) % 16 == 0);
    const int occ = spec::walk_occupancy((int)ldt, false);
    if (occ < 1) return fail(SPEC_CUDA_ERROR, "spec_verify_greedy: kernel does not fit on this device");
    int S, SL;
    choose_slices(B, V, es, grid_for(occ, 1 << 30), spec::kMaxSlices, S, SL);
    A.S = S; A.SL = SL;
    A.S1 = max_slices_for(V);
    const int grid = grid_for(occ, B * S);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, Lw.zero_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_verify_greedy: memset");
    e = spec::walk_run(A, false, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_verify_greedy: launch");
    return SPEC_OK;
}

// ---------------------------------------------------------------------------
// tree build
// ---------------------------------------------------------------------------
static Layout build_layout(int B, int L, int V, int budget) {
    return make_layout(B, static_cast<long long>(B) * (L + 1), budget > 1 ? budget - 1 : 1,
                       spec::build_extra_bytes(budget, L), max_slices_for(V));
}

size_t spec_tree_build_workspace_size(int B, int L, int V, int budget) {
    if (B < 0 || L < 0 || L > 16 || V < 1 || budget < 1 || budget > 256) return 0;
    return build_layout(B, L, V, budget).total;
}

spec_status spec_tree_build(
    const float* q, int64_t q_batch_stride, int64_t q_row_stride,
    int B, int L, int V, int budget,
    int32_t* token, int32_t* parent, int32_t* depth, double* score,
    uint64_t* anc_mask, int32_t* num_nodes, int32_t* status,
    void* ws, size_t ws_bytes, void* stream) {
    if (B < 0 || L < 0 || V < 1 || budget < 1)
        return fail(SPEC_INVALID_ARG, "spec_tree_build: need B >= 0, L >= 0, V >= 1, budget >= 1");
    if (L > 16 || budget > 256) return fail(SPEC_UNSUPPORTED, "spec_tree_build: L <= 16 and budget <= 256");
    if (B > spec::kMaxRecB) return fail(SPEC_UNSUPPORTED, "spec_tree_build: B > %d", spec::kMaxRecB);
    if (B == 0) return SPEC_OK;
    if (!token || !parent || !depth || !score || !anc_mask || !num_nodes || !status || !ws || (L > 0 && !q))
        return fail(SPEC_INVALID_ARG, "spec_tree_build: null pointer argument");
    if (q_row_stride < V || q_batch_stride < 0)
        return fail(SPEC_INVALID_ARG, "spec_tree_build: row stride must be >= V");
    const Layout Lw = build_layout(B, L, V, budget);
    if (ws_bytes < Lw.total)
        return fail(SPEC_INVALID_ARG, "spec_tree_build: workspace too small (%zu < %zu)", ws_bytes, Lw.total);
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "spec_tree_build: workspace must be 16-byte aligned");
    spec::BuildArgs A{};
    A.q = q; A.q_bs = q_batch_stride; A.q_rs = q_row_stride;
    A.B = B; A.L = L; A.V = V; A.N = budget; A.M = budget - 1;
    A.token = token; A.parent = parent; A.depth = depth; A.score = score;
    A.anc_mask = reinterpret_cast<unsigned long long*>(anc_mask);
    A.num_nodes = num_nodes; A.status = status;
    A.W = make_ws(ws, Lw);
    A.cap_p = budget > 1 ? budget - 1 : 1;
    A.tma_q = q && aligned16(q) && (q_row_stride * 4) % 16 == 0 && (q_batch_stride * 4) % 16 == 0;
    const int occ = spec::build_occupancy(budget, L);
    if (occ < 1) return fail(SPEC_CUDA_ERROR, "spec_tree_build: kernel does not fit on this device");
    int S, SL;
    choose_slices(B, V, 4, grid_for(occ, 1 << 30), spec::build_max_slices(budget, L), S, SL);
    A.S = S; A.SL = SL;
    A.S1 = spec::build_max_slices(budget, L) < max_slices_for(V) ? spec::build_max_slices(budget, L) : max_slices_for(V);
    const int grid = grid_for(occ, B * S);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, Lw.zero_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_tree_build: memset");
    e = spec::build_run(A, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_tree_build: launch");
    return SPEC_OK;
}

// ---------------------------------------------------------------------------
// tree walk
// ---------------------------------------------------------------------------
static Layout tree_layout(int B, int N, int V) {
    return make_layout(B, static_cast<long long>(B) * (N + 1), 0, 0, max_slices_for(V));
}

size_t spec_verify_tree_workspace_size(int B, int N, int V) {
    if (B < 0 || N < 1 || V < 1) return 0;
    return tree_layout(B, N, V).total;
}

spec_status spec_verify_tree(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* token, const int32_t* parent, const int32_t* num_nodes,
    int B, int N, int V, int max_depth,
    int32_t* path_nodes, int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
    void* ws, size_t ws_bytes, void* stream) {
    if (B < 0 || N < 1 || V < 1 || max_depth < 0)
        return fail(SPEC_INVALID_ARG, "spec_verify_tree: need B >= 0, N >= 1, V >= 1, max_depth >= 0");
    if (!valid_dtype(ldt)) return fail(SPEC_INVALID_ARG, "spec_verify_tree: unknown logits dtype");
    if (B > spec::kMaxRecB || N > spec::kMaxRecRow + 1)
        return fail(SPEC_UNSUPPORTED, "spec_verify_tree: B > %d or N > %d", spec::kMaxRecB, spec::kMaxRecRow + 1);
    if (B == 0) return SPEC_OK;
    if (!logits || !token || !parent || !num_nodes || !path_nodes || !out_tokens || !num_accepted || !status || !ws)
        return fail(SPEC_INVALID_ARG, "spec_verify_tree: null pointer argument");
    if (l_row_stride < V || l_batch_stride < 0)
        return fail(SPEC_INVALID_ARG, "spec_verify_tree: row stride must be >= V");
    const Layout Lw = tree_layout(B, N, V);
    if (ws_bytes < Lw.total)
        return fail(SPEC_INVALID_ARG, "spec_verify_tree: workspace too small (%zu < %zu)", ws_bytes, Lw.total);
    if (!aligned16(ws)) return fail(SPEC_INVALID_ARG, "spec_verify_tree: workspace must be 16-byte aligned");
    const int es = esize_of(ldt);
    spec::WalkArgs A{};
    A.logits = logits; A.l_bs = l_batch_stride; A.l_rs = l_row_stride;
    A.B = B; A.K = 0; A.V = V; A.ldt = (int)ldt;
    A.token = token; A.parent = parent; A.num_nodes = num_nodes; A.N = N; A.L = max_depth;
    A.path_nodes = path_nodes; A.out_tokens = out_tokens; A.num_accepted = num_accepted; A.status = status;
    A.W = make_ws(ws, Lw);
    A.tma_l = aligned16(logits) && (l_row_stride * es) % 16 == 0 && (l_batch_stride * es) % 16 == 0;
    const int occ = spec::walk_occupancy((int)ldt, true);
    if (occ < 1) return fail(SPEC_CUDA_ERROR, "spec_verify_tree: kernel does not fit on this device");
    int S, SL;
    choose_slices(B, V, es, grid_for(occ, 1 << 30), spec::kMaxSlices, S, SL);
    A.S = S; A.SL = SL;
    A.S1 = max_slices_for(V);
    const int grid = grid_for(occ, B * S);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, Lw.zero_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_verify_tree: memset");
    e = spec::walk_run(A, true, grid, st);
    if (e != cudaSuccess) return cuda_fail(e, "spec_verify_tree: launch");
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
    cudaError_t e = spec::adaptive_run(conf, B, Kmax, a, b, k_out, surv, exp_adv, l_row_off, q_row_off,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "spec_adaptive_len: launch");
    return SPEC_OK;
}

}  // extern "C"
