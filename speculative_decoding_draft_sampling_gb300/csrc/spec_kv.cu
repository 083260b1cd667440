// spec_kv.cu -- accepted-path KV compaction.
//
// [SD-survey] = "大模型投机解码：Medusa、MTP、EAGLE、DFlash、DDTree 与 DSpark"
// (Speculative decoding for LLMs: Medusa, MTP, EAGLE, DFlash, DDTree and
// DSpark), chzhyang.github.io, §5 "DDTree": after verification only the
// accepted path's KV is kept.  The tree's forward pass wrote one KV row per
// tree node; the root and the accepted nodes' rows move, in depth order, to
// the request's next cache positions, in every plane (a layer's keys or
// values).
//
// A gather bound by HBM bandwidth: one warp per (plane, request, path
// position); rows move in 16-byte vectors, four per lane in flight (all
// loads issued before the stores), or in 4-byte words / bytes when the
// layout is not 16-byte aligned.
#include "spec_chain.cuh"

namespace spec {


template <int kW>
__device__ __forceinline__ void copy_row(unsigned char* to, const unsigned char* from, long long bytes, int lane) {
    if constexpr (kW == 16) {
        const uint4* s = reinterpret_cast<const uint4*>(from);
        uint4* d = reinterpret_cast<uint4*>(to);
        const long long nv = bytes >> 4;
        for (long long v0 = lane; v0 < nv; v0 += 128) {
            uint4 r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (v0 + 32 * q < nv) r[q] = __ldcs(s + v0 + 32 * q);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (v0 + 32 * q < nv) __stcs(d + v0 + 32 * q, r[q]);
        }
    } else if constexpr (kW == 4) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(from);
        uint32_t* d = reinterpret_cast<uint32_t*>(to);
        for (long long v = lane; v < (bytes >> 2); v += 32) d[v] = s[v];
    } else {
        for (long long v = lane; v < bytes; v += 32) to[v] = from[v];
    }
}

template <int kW>
__global__ void __launch_bounds__(256) kv_compact_kernel(const KvArgs A) {
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const long long total = static_cast<long long>(A.P) * A.B * A.W;
    for (long long r = warp; r < total; r += nwarps) {
        const int j = static_cast<int>(r % A.W);
        const long long pb = r / A.W;
        const int b = static_cast<int>(pb % A.B);
        const int p = static_cast<int>(pb / A.B);
        if (j > A.num_accepted[b]) continue;
        const int node = A.path_nodes[static_cast<long long>(b) * A.W + j];
        if (node < 0 || node >= A.N) continue;
        const long long pos = (A.dst_pos ? A.dst_pos[b] : 0) + j;
        const unsigned char* from = A.src + p * A.s_plane + b * A.s_batch + node * A.s_row;
        unsigned char* to = A.dst + p * A.d_plane + b * A.d_batch + pos * A.d_row;
        copy_row<kW>(to, from, A.row_bytes, lane);
    }
}

cudaError_t kv_compact_run(const KvArgs& A, int sms, cudaStream_t st) {
    const long long rows = static_cast<long long>(A.P) * A.B * A.W;
    long long blocks = (rows + 7) / 8;                     // eight warps a block
    const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (A.width == 16) kv_compact_kernel<16><<<grid, 256, 0, st>>>(A);
    else if (A.width == 4) kv_compact_kernel<4><<<grid, 256, 0, st>>>(A);
    else kv_compact_kernel<1><<<grid, 256, 0, st>>>(A);
    return cudaGetLastError();
}

}  // namespace spec
