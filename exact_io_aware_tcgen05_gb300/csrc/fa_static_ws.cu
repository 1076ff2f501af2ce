// fa_static_ws.cu -- fa_bwd_static_workspace: the backward pass without any
// caller-provided or library-allocated device workspace.
//
// Some callers cannot call cudaMalloc at the point where they run the
// backward pass: code running inside a framework whose allocator owns all
// device memory, plugins that may not allocate behind their host's back, and
// code paths that must not allocate at all because an allocation would
// synchronise the device or could fail at an awkward time.  This entry point
// serves them: its scratch (fa_bwd's workspace: the fp32 row statistics
// D_i = dO_i . O_i and, for the fused backward, the fp32 dQ accumulator and its
// turn counters) lives in a fixed-size array below, which the library's image
// carries on every GPU that loads the library, for as long as the process lives.
//
// The array is shared by every call on a device and keeps what the last call
// left in it.  Nothing in it has to start at zero: the backward pass writes
// every D_i before any kernel reads it, zeroes the turn counters in its first
// kernel, and stores (not adds) each accumulator tile's first contribution.  Calls whose work overlaps on the GPU
// (different streams, or different host threads on one device) race on the
// array and must be serialised by the caller.
#include "../../include/fa.h"
#include "fa_kernels.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[FA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_ptr[kMaxDevices] = {nullptr};
unsigned long long g_ws_ctx[kMaxDevices] = {0};
// Device address of the array on the current device (host code cannot use the
// array's name as a device address).  Looked up on a device's first call and
// again whenever the device's context has changed since (a cudaDeviceReset
// destroys the context the cached address belonged to).
fa_status static_workspace_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fa::report_error(FA_ERR_CUDA, "fa_bwd_static_workspace: no usable current device (%s)",
                                cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long ctx = fa::current_context_id();
    if (!g_ws_ptr[dev] || ctx == 0 || ctx != g_ws_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess || !p)
            return fa::report_error(FA_ERR_CUDA,
                                    "fa_bwd_static_workspace: cudaGetSymbolAddress failed on "
                                    "device %d (%s)",
                                    dev, cudaGetErrorString(e));
        g_ws_ptr[dev] = p;
        g_ws_ctx[dev] = fa::current_context_id();
    }
    *out = g_ws_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_static_workspace(const void* q, const void* k, const void* v,
                                             const void* o, const float* lse, const void* dout,
                                             void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                             int N, int d, int causal, int window,
                                             const int* cu_seqlens, int total_tokens, float scale,
                                             cudaStream_t stream) {
    // the least workspace fa_bwd accepts (its split backward); fa_bwd itself picks
    // the fused backward when the array also holds that one's dQ accumulator
    const size_t need =
        fa_bwd_workspace_size_min(B, Hq, Hkv, N, d, cu_seqlens ? total_tokens : 0);
    if (need > static_cast<size_t>(FA_STATIC_WORKSPACE_BYTES)) {
        // a rejected call uses up timing events armed for it, as fa_bwd's own
        // argument errors do
        fa_set_launch_events(nullptr, 0);
        return fa::report_error(FA_ERR_WORKSPACE,
                                "fa_bwd_static_workspace: these sizes need %zu bytes of scratch, "
                                "more than the %d-byte static array; use fa_bwd with a "
                                "caller-provided workspace",
                                need, FA_STATIC_WORKSPACE_BYTES);
    }
    void* ws = nullptr;
    const fa_status st = static_workspace_address(&ws);
    if (st != FA_OK) return st;
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, window, cu_seqlens,
                  total_tokens, scale, ws, FA_STATIC_WORKSPACE_BYTES, stream);
}
