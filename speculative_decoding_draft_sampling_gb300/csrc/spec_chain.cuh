// spec_chain.cuh -- argument blocks of the engine kernels and the host-side
// launch functions each translation unit provides.
#pragma once

#include "spec_engine.cuh"

namespace spec {

struct ChainArgs {
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
    const int* k_per_req;
    const int* l_row_off;
    const int* q_row_off;
    int* out_tokens;
    int* num_accepted;
    int* status;
    float* diag;
    Workspace W;
    int S, SL, cap_p;              // slices of a first row and their length
    int S1;                        // most slices of a pushed row
    int tma_l, tma_q;
};

struct WalkArgs {                  // greedy verify and tree walk
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
    Workspace W;
    int S, SL;                     // slices of a first row and their length
    int S1;                        // most slices of a pushed row
    int tma_l;
};

struct BuildArgs {
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
    Workspace W;
    int S, SL, cap_p;              // slices of a first row and their length
    int S1;                        // most slices of a pushed row
    int tma_q;
};

// slices of a task and their length: first rows take the call's, pushed
// rows carry their own in the kind word
template <class Args>
__device__ __forceinline__ int task_S(const Args& A, const Task& t) { return t.kind < 0 ? A.S : task_kind_S(t.kind); }
template <class Args>
__device__ __forceinline__ int task_SL(const Args& A, const Task& t) { return t.kind < 0 ? A.SL : task_kind_SL(t.kind); }

// chain
cudaError_t chain_run(const ChainArgs& A, int grid, cudaStream_t st);
size_t chain_smem(int ldt, bool topk);
int chain_occupancy(int ldt, bool topk);
// greedy / tree walk
cudaError_t walk_run(const WalkArgs& A, bool tree, int grid, cudaStream_t st);
int walk_occupancy(int ldt, bool tree);
// tree build
cudaError_t build_run(const BuildArgs& A, int grid, cudaStream_t st);
int build_occupancy(int N, int L);
size_t build_extra_bytes(int N, int L);
int build_max_slices(int N, int L);
// error text for spec_last_error() from outside the API file
void set_last_error(const char* msg);
// adaptive length
cudaError_t adaptive_run(const float* conf, int B, int Kmax, float a, float b, int* k_out, double* surv,
                         double* exp_adv, int* l_off, int* q_off, cudaStream_t st);

}  // namespace spec
