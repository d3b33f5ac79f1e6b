// awq_search_scale_noalloc: the alpha search with its scratch memory in a
// fixed, library-owned device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory: plug-ins hosted by an
// inference server or framework that owns the whole device memory pool and
// does not let its extensions allocate, and latency-critical loops that rule
// out cudaMalloc because it can synchronise the device.  This entry point
// needs no allocation from anyone: the caller passes only inputs and outputs,
// and the scratch lives in g_search_scratch below.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds its AWQ_SEARCH_NOALLOC_SCRATCH_BYTES until the process
// exits.  In host code its name is only a host-side stand-in: the device
// address is looked up with cudaGetSymbolAddress on the first call of this
// entry point on a device (with that device current; make that first call
// before any stream capture), again whenever the device's current context
// has changed since (e.g. after cudaDeviceReset), and passed to the kernels
// as their workspace.  All calls share the one array and it keeps the
// last call's contents; nothing in it has to start at zero, because every
// scratch element a call reads is written earlier by the same call.  Calls
// that overlap on the GPU (for example on two streams) race on the array.
#include <mutex>
#include <stdio.h>

#include "awq.h"
#include "common.cuh"
#include "kernels.cuh"

namespace awq {
awq_status report_error(awq_status code, const char* msg);
}

namespace {

constexpr size_t kScratchBytes = AWQ_SEARCH_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_search_scratch[kScratchBytes];

// The array's device address, per device, for the context it was looked up
// in: a symbol address belongs to one CUDA context, so a call made in another
// context (the new primary context after cudaDeviceReset, or a context the
// caller created) looks it up again instead of using a stale address.
constexpr int kMaxDevices = 64;
struct ScratchAddr {
    void* ptr = nullptr;
    unsigned long long ctx_id = 0;
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

}  // namespace

extern "C" awq_status awq_search_scale_noalloc(const uint16_t* W, int64_t N, int64_t K,
                                               int64_t ldw, const uint16_t* Xcal, int64_t T,
                                               int64_t ldx, const double* mean_abs,
                                               const double* alphas, int n_alpha, int group,
                                               float* s_out, double* mse_out, int32_t* best_idx,
                                               float* s_alpha_out, awq_stream_t stream) {
    // the sizes that define the scratch need are checked first, so that a bad
    // argument is reported as such and not as a scratch shortage
    if (N <= 0 || K <= 0 || T <= 0 || n_alpha < 1 || n_alpha > AWQ_MAX_ALPHAS)
        return awq::report_error(AWQ_ERR_INVALID_ARG,
                                 "search_scale_noalloc: sizes must be positive, 1 <= n_alpha <= 64");
    const size_t need = awq_search_workspace_size(N, K, T, n_alpha);
    if (need > kScratchBytes) {
        static thread_local char msg[192];
        snprintf(msg, sizeof msg,
                 "search_scale_noalloc: this problem needs %zu bytes of scratch, more than the "
                 "%zu MiB the library holds; use awq_search_scale with a caller workspace",
                 need, kScratchBytes >> 20);
        return awq::report_error(AWQ_ERR_WORKSPACE, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return awq::report_error(AWQ_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return awq::report_error(AWQ_ERR_DEVICE, "search_scale_noalloc: device index out of range");
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        ScratchAddr& a = g_scratch[dev];
        const unsigned long long ctx = awq::context_id();
        if (!a.ptr || (ctx != 0 && ctx != a.ctx_id)) {
            a.ptr = nullptr;
            e = cudaGetSymbolAddress(&a.ptr, g_search_scratch);
            if (e != cudaSuccess) {
                a.ptr = nullptr;
                cudaGetLastError();
                return awq::report_error(AWQ_ERR_CUDA,
                                         "search_scale_noalloc: cudaGetSymbolAddress failed");
            }
            a.ctx_id = awq::context_id();
        }
        scratch = a.ptr;
    }
    return awq_search_scale(W, N, K, ldw, Xcal, T, ldx, mean_abs, alphas, n_alpha, group, s_out,
                            mse_out, best_idx, s_alpha_out, scratch, kScratchBytes, stream);
}
