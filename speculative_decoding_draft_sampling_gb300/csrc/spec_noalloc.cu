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

constexpr size_t kStaticWorkspaceBytes = size_t(64) << 10;   // 64 KiB, held by every GPU that loads the library

// Device memory; in host code this name is only a stand-in, never a usable
// device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};
void* g_ws_ctx[kMaxDevices] = {};   // the context the address belongs to

// The current CUDA context, through the driver entry point the runtime
// resolves (no link-time dependency on the driver library); null if none.
typedef int (*CtxGetCurrentFn)(void**);
void* current_context() {
    static CtxGetCurrentFn fn = nullptr;
    static bool looked = false;
    if (!looked) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        looked = true;
    }
    void* ctx = nullptr;
    if (!fn || fn(&ctx) != 0) return nullptr;
    return ctx;
}

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
                             "64 KiB static one; use spec_verify_greedy with a caller-provided workspace");
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
        // First call on this device (made current): look up the array's
        // device address.  The address belongs to the context the library's
        // module was loaded into; after a device reset the device has a new
        // context, so a changed context handle repeats the look-up.
        std::lock_guard<std::mutex> lk(g_mu);
        void* ctx = current_context();
        if (!g_ws_addr[dev] || ctx == nullptr || ctx != g_ws_ctx[dev]) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_static_workspace);
            if (e != cudaSuccess) {
                g_ws_addr[dev] = nullptr;
                g_ws_ctx[dev] = nullptr;
                spec::set_last_error("spec_verify_greedy_static: cudaGetSymbolAddress failed");
                return SPEC_CUDA_ERROR;
            }
            g_ws_addr[dev] = addr;
            g_ws_ctx[dev] = current_context();
        }
        ws = g_ws_addr[dev];
    }
    return spec_verify_greedy(logits, ldt, l_batch_stride, l_row_stride, draft, B, K, V, k_per_req, l_row_off,
                              out_tokens, num_accepted, status, ws, kStaticWorkspaceBytes, stream);
}
