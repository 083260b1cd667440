// spec_chain.cuh -- argument blocks of the engine kernels and the host-side
// launch helpers each translation unit provides.
#pragma once

#include "spec_engine.cuh"

namespace spec {

struct ChainArgs {
    EngArgs E;
    const void* logits;
    long long l_bs, l_rs;          // element strides
    const float* q;
    long long q_bs, q_rs;
    const int* draft;
    const float* uniforms;
    int B, K, V, ldt;
    float c2;                      // log2(e) / T, fp32
    double Td;                     // T
    int top_k;
    const int* k_per_req;          // per-request verify length (NULL: K for all)
    const int* l_row_off;          // packed rows (NULL with k_per_req: dense rows, capped at k_b)
    const int* q_row_off;
    int* out_tokens;
    int* num_accepted;
    int* status;
    float* diag;
    int cap_p;                     // candidate keys a slice may report
    int tma_l, tma_q;
    // stochastic tree walk: rows are tree nodes ([B, N, V] logits), the
    // uniforms are [B, L+1] (one per depth), outputs are [B, L+1]
    int tree;
    const int* t_token;
    const int* t_parent;
    const int* t_nn;
    int N, L;
    int* path_nodes;
};

// lowest child of node `cur` of request b whose token is t (-1: none), all
// lanes of a warp
__device__ __forceinline__ int find_child_w(const int* token, const int* parent, const int* num_nodes, int N, int b,
                                            int cur, int t) {
    const int l = threadIdx.x & 31;
    int child = 0x7fffffff;
    int nn = num_nodes[b];
    nn = nn < N ? nn : N;
    const int* par = parent + static_cast<long long>(b) * N;
    const int* tok = token + static_cast<long long>(b) * N;
    for (int c = l; c < nn; c += 32)
        if (par[c] == cur && tok[c] == t) child = min(child, c);
    child = static_cast<int>(warp_min_u32(static_cast<uint32_t>(child)));
    return child == 0x7fffffff ? -1 : child;
}

struct WalkArgs {                  // greedy verify and tree walks
    EngArgs E;
    const void* logits;
    long long l_bs, l_rs;
    int B, K, V, ldt;
    const int* draft;              // greedy
    const int* k_per_req;
    const int* l_row_off;
    const int* token;              // tree
    const int* parent;
    const int* num_nodes;
    int N, L;
    int* path_nodes;
    int* out_tokens;
    int* num_accepted;
    int* status;
    // stochastic tree walk
    const float* uniforms;         // [B, L+1] (NULL: greedy walk)
    float c2;
    int top_k;
    float* diag;                   // NULL or [B, L+1, 2]: p(token), Z per walked node
    int tma_l;
};

struct BuildArgs {
    EngArgs E;
    const float* q;
    long long q_bs, q_rs;
    int B, L, V, N, M;
    int* token;
    int* parent;
    int* depth;
    double* score;
    unsigned long long* anc_mask;
    int* num_nodes;
    int* status;
    int cap_p;                     // keys a slice may report (M)
    int tma_q;
};

// EAGLE-2 expansion rows: unit u = b * F + f is frontier slot f of request
// b; its q row is base.q + b * base.q_bs + f * base.q_rs.  Each unit's top-K2
// (base.M) children go to the unit's workspace extra: EagleRowHdr, then K2
// tokens, then K2 probabilities.
struct EagleArgs {
    BuildArgs base;                // q, strides, B, V, M = K2, cap_p, tma_q, E
    int F, G;
    const int* front_in;           // [B, F]
    const int* num_front_in;       // [B]
    const int* num_gen;            // [B]
    const double* score;           // [B, G] node scores
    const int* depth;              // [B, G] node depths
};
struct EagleRowHdr {
    int n;                         // children found; -1: no row (slot past the frontier); -2: bad node id
    int bad;                       // the row held a NaN or +inf
    int node;                      // the frontier node the row belongs to (n >= 0)
    int depth;                     // that node's depth
    double score;                  // and its score
    double pad;
};
size_t eagle_row_extra_bytes(int K2);
const void* eagle_rows_kernel_ptr();
size_t eagle_rows_smem(int C, int own, int part_bytes, int stages, int chunk);
// the grow step (one CTA per request) and the rerank
struct EagleGrowArgs {
    const unsigned char* rows;     // workspace extras of the row units
    long long row_stride;          // bytes between units
    int B, F, K2, Fn, G;
    int* token; int* parent; int* depth; double* score; int* num_gen;
    const int* front_in; const int* num_front_in;
    int* front_out; int* num_front_out; int* status;
};
cudaError_t eagle_grow_run(const EagleGrowArgs& A, cudaStream_t st);
struct EagleRerankArgs {
    const int* token; const int* parent; const int* depth; const double* score; const int* num_gen;
    int B, G, N;
    int* out_token; int* out_parent; int* out_depth; double* out_score;
    unsigned long long* anc_mask; int* num_nodes; int* status;
};
cudaError_t eagle_rerank_run(const EagleRerankArgs& A, cudaStream_t st);
// chain
const void* chain_kernel_ptr(int ldt, bool topk);
size_t chain_smem(int C, int own, int part_bytes, int stages, int chunk);
int chain_part_bytes(int top_k, int cap_p);
// greedy / tree walk
const void* walk_kernel_ptr(int ldt, int mode);   // mode 0 greedy, 1 tree, 2 stochastic tree
size_t walk_smem(int C, int own, int part_bytes, int stages, int chunk);
int walk_part_bytes();
// tree build
const void* build_kernel_ptr();
size_t build_smem(int C, int own, int part_bytes, int stages, int chunk, int N, int L);
int build_part_bytes(int M);
size_t build_extra_bytes(int N, int L);
// accepted-path KV compaction
struct KvArgs {
    const unsigned char* src;
    long long s_plane, s_batch, s_row;    // bytes
    unsigned char* dst;
    long long d_plane, d_batch, d_row;    // bytes
    int P, B, N, W;
    long long row_bytes;
    const int* path_nodes;                // [B, W]
    const int* num_accepted;              // [B]
    const int* dst_pos;                   // [B] or null
    int width;                            // 16, 4 or 1: the copy unit the layout allows
};
cudaError_t kv_compact_run(const KvArgs& A, int sms, cudaStream_t st);
// error text for spec_last_error() from outside the API file
void set_last_error(const char* msg);
// adaptive length
cudaError_t adaptive_run(const float* conf, int B, int Kmax, float a, float b, const double* cost, int* k_out,
                         double* surv, double* exp_adv, int* l_off, int* q_off, cudaStream_t st);

}  // namespace spec
