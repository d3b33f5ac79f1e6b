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
// address is looked up once per device with cudaGetSymbolAddress, on the
// first call of this entry point on that device with that device current
// (make that first call before any stream capture), and passed to the
// kernels as their workspace.  All calls share the one array and it keeps the
// last call's contents; nothing in it has to start at zero, because every
// scratch element a call reads is written earlier by the same call.  Calls
// that overlap on the GPU (for example on two streams) race on the array.
#include <mutex>

#include "awq.h"
#include "kernels.cuh"

namespace awq {
awq_status report_error(awq_status code, const char* msg);
}

namespace {

constexpr size_t kScratchBytes = AWQ_SEARCH_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_search_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

}  // namespace

extern "C" awq_status awq_search_scale_noalloc(const uint16_t* W, int64_t N, int64_t K,
                                               int64_t ldw, const uint16_t* Xcal, int64_t T,
                                               int64_t ldx, const double* mean_abs,
                                               const double* alphas, int n_alpha, int group,
                                               float* s_out, double* mse_out, int32_t* best_idx,
                                               float* s_alpha_out, awq_stream_t stream) {
    const size_t need = awq_search_workspace_size(N, K, T, n_alpha);
    if (need > kScratchBytes)
        return awq::report_error(AWQ_ERR_WORKSPACE,
                                 "search_scale_noalloc: this problem needs more scratch than the "
                                 "16 MiB (AWQ_SEARCH_NOALLOC_SCRATCH_BYTES) the library holds; "
                                 "use awq_search_scale with a caller workspace");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return awq::report_error(AWQ_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return awq::report_error(AWQ_ERR_DEVICE, "search_scale_noalloc: device index out of range");
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            e = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_search_scratch);
            if (e != cudaSuccess) {
                g_scratch_ptr[dev] = nullptr;
                cudaGetLastError();
                return awq::report_error(AWQ_ERR_CUDA,
                                         "search_scale_noalloc: cudaGetSymbolAddress failed");
            }
        }
        scratch = g_scratch_ptr[dev];
    }
    return awq_search_scale(W, N, K, ldw, Xcal, T, ldx, mean_abs, alphas, n_alpha, group, s_out,
                            mse_out, best_idx, s_alpha_out, scratch, kScratchBytes, stream);
}
