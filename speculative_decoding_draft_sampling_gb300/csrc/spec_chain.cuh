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

// chain
const void* chain_kernel_ptr(int ldt, bool topk);
size_t chain_smem(int C, int own, int part_bytes, int stages);
int chain_part_bytes(int top_k, int cap_p);
// greedy / tree walk
const void* walk_kernel_ptr(int ldt, int mode);   // mode 0 greedy, 1 tree, 2 stochastic tree
size_t walk_smem(int C, int own, int part_bytes, int stages);
int walk_part_bytes();
// tree build
const void* build_kernel_ptr();
size_t build_smem(int C, int own, int part_bytes, int stages, int N, int L);
int build_part_bytes(int M);
size_t build_extra_bytes(int N, int L);
// error text for spec_last_error() from outside the API file
void set_last_error(const char* msg);
// adaptive length
cudaError_t adaptive_run(const float* conf, int B, int Kmax, float a, float b, const double* cost, int* k_out,
                         double* surv, double* exp_adv, int* l_off, int* q_off, cudaStream_t st);

}  // namespace spec
