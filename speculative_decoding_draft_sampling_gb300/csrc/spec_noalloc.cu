// spec_noalloc.cu -- greedy verification for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they verify: code running inside a host callback or an
// allocator-free runtime, plugins handed raw buffers by a host engine that
// owns every allocation, or real-time loops that forbid allocation after
// start-up.  spec_verify_greedy needs a scratch workspace; this variant
// takes it from a fixed array in device global memory that the library
// reserves when it is loaded, so the caller passes only inputs and outputs.
//
// The array is shared by every call on a device and keeps the previous
// call's contents; the verification itself zeroes the queue counters it
// needs at the start of each call.  Two calls whose GPU work overlaps (two
// streams, or two host threads on one device) race on it.
#include <mutex>

#include "../../include/spec_verify.h"
#include "spec_chain.cuh"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(8) << 20;   // 8 MiB, held by every GPU that loads the library

// Device memory; in host code this name is only a stand-in, never a usable
// device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};

}  // namespace

extern "C" spec_status spec_verify_greedy_static(
    const void* logits, spec_dtype ldt, int64_t l_batch_stride, int64_t l_row_stride,
    const int32_t* draft, int B, int K, int V,
    const int32_t* k_per_req, const int32_t* l_row_off,
    int32_t* out_tokens, int32_t* num_accepted, int32_t* status, void* stream) {
    if (B < 0 || K < 0 || V < 1) {
        spec::set_last_error("spec_verify_greedy_static: need B >= 0, K >= 0, V >= 1");
        return SPEC_INVALID_ARG;
    }
    const size_t need = spec_verify_greedy_workspace_size(B, K, V);
    if (need > kStaticWorkspaceBytes) {
        spec::set_last_error("spec_verify_greedy_static: this batch needs a larger workspace than the "
                             "8 MiB static one; use spec_verify_greedy with a caller-provided workspace");
        return SPEC_INVALID_ARG;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        spec::set_last_error("spec_verify_greedy_static: no usable current device");
        return SPEC_CUDA_ERROR;
    }
    void* ws = nullptr;
    {
        // first call on this device (made current): look up the array's device address once
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_ws_addr[dev]) {
            e = cudaGetSymbolAddress(&g_ws_addr[dev], g_static_workspace);
            if (e != cudaSuccess) {
                g_ws_addr[dev] = nullptr;
                spec::set_last_error("spec_verify_greedy_static: cudaGetSymbolAddress failed");
                return SPEC_CUDA_ERROR;
            }
        }
        ws = g_ws_addr[dev];
    }
    return spec_verify_greedy(logits, ldt, l_batch_stride, l_row_stride, draft, B, K, V, k_per_req, l_row_off,
                              out_tokens, num_accepted, status, ws, kStaticWorkspaceBytes, stream);
}
