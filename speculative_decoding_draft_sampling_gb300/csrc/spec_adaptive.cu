// spec_adaptive.cu -- DSpark verify length.
//
// [SD-survey] = "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
// (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash, DDTree and
// DSpark), chzhyang.github.io, §5 "DSpark": with conditional confidences c_i,
// the prefix survives to position j with probability s_j = prod_{i<=j} c_i,
// and verifying k positions advances 1 + sum_{j<=k} s_j tokens in
// expectation.  Each request takes the k in [0, Kmax] with the largest
// advance per unit cost a + b*k (the question the page poses: is one more
// position worth its cost?); ties go to the smaller k.  The ragged row
// offsets of the verify that follows (SGLang's "compact" mode, §9) are the
// exclusive scans of k+1 (logits rows) and k (draft rows).
//
// Arithmetic is fp64 with explicit round-to-nearest intrinsics, so no
// multiply-add is fused and the sequence of roundings is the plain one:
// s = s*c_j; E = E + s; ratio = E / (a + b*j).  With a cost table (§9: the
// per-deployment profile of what verifying k positions costs) the ratio is
// E / cost[j] instead.
#include "spec_chain.cuh"

namespace spec {

constexpr int kAdaptThreads = 256;

__global__ void __launch_bounds__(kAdaptThreads) adaptive_kernel(const float* __restrict__ conf, int B, int Kmax,
                                                                  double a, double bc,
                                                                  const double* __restrict__ cost,
                                                                  int* __restrict__ k_out,
                                                                  double* __restrict__ surv,
                                                                  double* __restrict__ exp_adv,
                                                                  int* __restrict__ l_off, int* __restrict__ q_off) {
    __shared__ int wsum[2][kAdaptThreads / 32];
    __shared__ int carry[2];
    if (threadIdx.x == 0) { carry[0] = 0; carry[1] = 0; }
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int b0 = 0; b0 < B; b0 += kAdaptThreads) {
        const int r = b0 + threadIdx.x;
        int kbest = 0;
        if (r < B) {
            double s = 1.0, E = 1.0;
            double best = __ddiv_rn(1.0, cost ? cost[0] : __dadd_rn(a, __dmul_rn(bc, 0.0)));
            double bestE = 1.0;
            for (int j = 1; j <= Kmax; ++j) {
                s = __dmul_rn(s, static_cast<double>(conf[static_cast<long long>(r) * Kmax + (j - 1)]));
                if (surv) surv[static_cast<long long>(r) * Kmax + (j - 1)] = s;
                E = __dadd_rn(E, s);
                const double ratio =
                    __ddiv_rn(E, cost ? cost[j] : __dadd_rn(a, __dmul_rn(bc, static_cast<double>(j))));
                if (ratio > best) { best = ratio; kbest = j; bestE = E; }
            }
            k_out[r] = kbest;
            if (exp_adv) exp_adv[r] = bestE;
        }
        // exclusive scans of (k+1) and k over this chunk, plus the running carry
        int v0 = r < B ? kbest + 1 : 0, v1 = r < B ? kbest : 0;
        int i0 = v0, i1 = v1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t0 = __shfl_up_sync(0xffffffffu, i0, o);
            const int t1 = __shfl_up_sync(0xffffffffu, i1, o);
            if (lane >= o) { i0 += t0; i1 += t1; }
        }
        if (lane == 31) { wsum[0][w] = i0; wsum[1][w] = i1; }
        __syncthreads();
        int base0 = carry[0], base1 = carry[1], tot0 = 0, tot1 = 0;
        for (int j = 0; j < kAdaptThreads / 32; ++j) {
            if (j < w) { base0 += wsum[0][j]; base1 += wsum[1][j]; }
            tot0 += wsum[0][j];
            tot1 += wsum[1][j];
        }
        if (r < B) {
            l_off[r] = base0 + i0 - v0;
            q_off[r] = base1 + i1 - v1;
        }
        __syncthreads();
        if (threadIdx.x == 0) { carry[0] += tot0; carry[1] += tot1; }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        l_off[B] = carry[0];
        q_off[B] = carry[1];
    }
}

cudaError_t adaptive_run(const float* conf, int B, int Kmax, float a, float b, const double* cost, int* k_out,
                         double* surv, double* exp_adv, int* l_off, int* q_off, cudaStream_t st) {
    adaptive_kernel<<<1, kAdaptThreads, 0, st>>>(conf, B, Kmax, static_cast<double>(a), static_cast<double>(b), cost,
                                                 k_out, surv, exp_adv, l_off, q_off);
    return cudaGetLastError();
}

}  // namespace spec
