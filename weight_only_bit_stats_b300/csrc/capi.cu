// C ABI of libawq_b300.so (declared in include/awq.h): argument checks,
// workspace carving, TMA descriptor creation and kernel dispatch.  The
// library allocates no device memory; every scratch buffer comes from the
// caller's workspace.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "awq.h"
#include "common.cuh"
#include "kernels.cuh"
#include "int3.cuh"

namespace {

// awq_set_weight_prefetch() state, read by every decode launch.
std::atomic<int> g_early_weights{0};

// Device status word (one per device that loads the library).
__device__ unsigned int g_awq_status;

thread_local const char* g_last_error = "no error";

// An NVTX range named after the C-ABI call it spans, so a profiler's
// timeline shows each call around its kernels.  Without a profiler attached
// the push and pop return at once.
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

constexpr int kMaxDevices = 64;
struct DevInfo {
    bool init = false;
    bool ok = false;
    int num_sms = 0;
    unsigned* status = nullptr;
    unsigned long long ctx_id = 0;   // context the status address belongs to
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

awq_status fail(awq_status code, const char* msg) {
    g_last_error = msg;
    return code;
}

awq_status cuda_fail(cudaError_t e) {
    g_last_error = cudaGetErrorString(e);
    return AWQ_ERR_CUDA;
}

// Driver entry points for the context id (the library links the runtime
// statically and reaches the driver through the runtime's entry-point query).
using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);
PfnCtxGetCurrent g_ctx_get_current = nullptr;
PfnCtxGetId g_ctx_get_id = nullptr;
std::once_flag g_ctx_once;

// Current device's info; checks compute capability 10.3 once per device and
// context, and looks the status word's address up again in a new context.
awq_status device_info(DevInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return fail(AWQ_ERR_DEVICE, "device index out of range");
    const unsigned long long ctx = awq::context_id();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo& d = g_dev[dev];
    if (!d.init || (ctx != 0 && ctx != d.ctx_id)) {
        d.init = true;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_awq_status);
        d.status = static_cast<unsigned*>(p);
        d.ok = (major == 10 && minor == 3 && e == cudaSuccess && d.status != nullptr);
        if (e != cudaSuccess) cudaGetLastError();
        d.ctx_id = awq::context_id();   // the lookup above made the context current
    }
    if (!d.ok) return fail(AWQ_ERR_DEVICE, "requires a compute capability 10.3 (sm_103a) device");
    *out = &d;
    return AWQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool load_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// Activations [rows, K] fp16 for the tensor-core kernels: 128-byte swizzled
// boxes of 64 k x kTcTokens rows.
awq_status make_act_map(CUtensorMap* map, const uint16_t* X, int64_t rows, int64_t K, int64_t ld) {
    if (!load_encoder()) return fail(AWQ_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)awq::kTcTokens};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(X), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(AWQ_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    return AWQ_OK;
}

// fp16 [rows, K] with boxes of 64 k x box_rows rows, 128-byte swizzle.
awq_status make_map_rows(CUtensorMap* map, const uint16_t* X, int64_t rows, int64_t K, int64_t ld,
                         int box_rows) {
    if (!load_encoder()) return fail(AWQ_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(X), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(AWQ_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    return AWQ_OK;
}

// Packed weights [N, K/8] uint32 as TMA boxes.  kQwDecode: unswizzled boxes
// of 48 words (three groups of 128 nibbles) x 16 rows for the decode kernel,
// landing as [16 rows][192 B].  kQwGemm: one group (16 words) x 128 rows for
// the tensor-core GEMM's producers, 64-byte swizzle (chunk j of row r lands
// at 64 r + 16 (j ^ ((r >> 1) & 3)), so a quarter warp reading one chunk of
// eight rows hits eight bank groups).  Matmuls are called on the same few
// weights over and over, so the encoded maps are kept in a small per-thread
// cache keyed on (address, N, K, kind) -- a map holds nothing else -- and
// the encode (driver work on the launch path) runs once per weight.
enum QwMapKind { kQwDecode = 0, kQwGemm = 1 };
struct QwMapEntry {
    const uint32_t* qw = nullptr;
    int64_t N = 0, K = 0;
    int kind = 0;
    CUtensorMap map;
};
constexpr int kQwMapCache = 16;
thread_local QwMapEntry t_qw_maps[kQwMapCache];
thread_local int t_qw_next = 0;

awq_status encode_qweight_map(CUtensorMap* map, const uint32_t* qw, int64_t N, int64_t K,
                              int kind);

awq_status make_qweight_map(CUtensorMap* map, const uint32_t* qw, int64_t N, int64_t K,
                            int kind = kQwDecode) {
    for (const QwMapEntry& e : t_qw_maps)
        if (e.qw == qw && e.N == N && e.K == K && e.kind == kind) {
            *map = e.map;
            return AWQ_OK;
        }
    awq_status s = encode_qweight_map(map, qw, N, K, kind);
    if (s) return s;
    QwMapEntry& e = t_qw_maps[t_qw_next];
    t_qw_next = (t_qw_next + 1) % kQwMapCache;
    e.qw = qw;
    e.N = N;
    e.K = K;
    e.kind = kind;
    e.map = *map;
    return AWQ_OK;
}

awq_status encode_qweight_map(CUtensorMap* map, const uint32_t* qw, int64_t N, int64_t K,
                              int kind) {
    if (!load_encoder()) return fail(AWQ_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {48, 16};
    CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (kind == kQwGemm) {
        box[0] = AWQ_GROUP / 8;
        box[1] = (cuuint32_t)awq::kTcRows;
        swz = CU_TENSOR_MAP_SWIZZLE_64B;
    }
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(qw), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(AWQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (qweight)");
    return AWQ_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace layout of awq_search_scale / awq_candidate_scales.
int current_num_sms();

// The Gram-route search's residual hand-over buffers: per CTA (at most one
// per SM) two [128 rows][512 columns] fp16 tiles.
size_t gram_exp_bytes(int num_sms) {
    return align256((size_t)num_sms * 2 * awq::kTcRows * awq::kSearchTokensPerItem * 2);
}

struct SearchWs {
    size_t s_alpha, inv_s, r, mm, partials, mse, total;
};
SearchWs search_ws(int64_t N, int64_t K, int64_t T, int n_alpha) {
    SearchWs w;
    const int64_t n_tiles = (N + awq::kTcRows - 1) / awq::kTcRows;
    const int64_t t_tiles = (T + awq::kSearchTokensPerItem - 1) / awq::kSearchTokensPerItem;
    size_t off = 0;
    w.s_alpha = off;  off += align256((size_t)n_alpha * K * 4);
    w.inv_s = off;    off += align256((size_t)n_alpha * K * 4);
    w.r = off;        off += align256((size_t)n_alpha * K * 8);
    w.mm = off;       off += align256((size_t)n_alpha * awq::cand_blocks(K) * 2 * 8);
    w.partials = off; off += align256((size_t)n_alpha * n_tiles * t_tiles * 4 * 8);
    w.mse = off;      off += align256((size_t)n_alpha * 8);
    w.total = off;
    return w;
}

}  // namespace

namespace awq {
// Lets other translation units of the library report an error message
// through awq_last_error_string().
awq_status report_error(awq_status code, const char* msg) { return fail(code, msg); }

unsigned long long context_id() {
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PfnCtxGetCurrent>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PfnCtxGetId>(fn);
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext c = nullptr;
    if (g_ctx_get_current(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    if (g_ctx_get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}
}  // namespace awq

extern "C" {

int awq_version(void) { return 100; }

awq_status awq_selftest_wait_timeout(int64_t limit_us, awq_stream_t stream) {
    const CallRange range("awq_selftest_wait_timeout");
    if (limit_us < 1 || limit_us > 1000000)
        return fail(AWQ_ERR_INVALID_ARG, "selftest_wait_timeout: limit must be 1 us .. 1 s");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaError_t e = awq::launch_wait_timeout_selftest((unsigned long long)limit_us * 1000ull,
                                                      d->status, (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

awq_status awq_set_weight_prefetch(int enable) {
    if (enable != 0 && enable != 1) return fail(AWQ_ERR_INVALID_ARG, "set_weight_prefetch: flag must be 0 or 1");
    g_early_weights.store(enable, std::memory_order_relaxed);
    return AWQ_OK;
}

const char* awq_last_error_string(void) { return g_last_error; }

awq_status awq_sync_status(awq_stream_t stream) {
    const CallRange range("awq_sync_status");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned v = 0;
    e = cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (v) {
        unsigned zero = 0;
        e = cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (v & awq::kStatusTimeout) return fail(AWQ_ERR_TIMEOUT, "a bounded device wait expired");
    if (v & awq::kStatusOverflow)
        return fail(AWQ_ERR_OVERFLOW, "an accumulated statistics sum reached 2^63 (too many tokens)");
    if (v & awq::kStatusNonFinite) return fail(AWQ_ERR_NONFINITE, "non-finite value on the device");
    return AWQ_OK;
}

awq_status awq_act_stats(const uint16_t* X, int64_t T, int64_t K, int64_t ldx, int accumulate,
                         int64_t* abs_sum_q24, awq_stream_t stream) {
    const CallRange range("awq_act_stats");
    if (T < 0 || K < 0 || (accumulate != 0 && accumulate != 1))
        return fail(AWQ_ERR_INVALID_ARG, "act_stats: negative size or bad accumulate flag");
    if (!abs_sum_q24 || (T > 0 && !X)) return fail(AWQ_ERR_INVALID_ARG, "act_stats: null pointer");
    if (K % 8 || ldx < K || ldx % 8) return fail(AWQ_ERR_SHAPE, "act_stats: K and ldx must be multiples of 8, ldx >= K");
    if (T >= (1LL << 23))
        return fail(AWQ_ERR_SHAPE, "act_stats: T must be below 2^23 tokens per call (exact int64 sums)");
    if ((X && !aligned16(X)) || (reinterpret_cast<uintptr_t>(abs_sum_q24) & 7u))
        return fail(AWQ_ERR_ALIGN, "act_stats: X must be 16-byte aligned");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (!accumulate && K > 0) e = cudaMemsetAsync(abs_sum_q24, 0, (size_t)K * 8, st);
    if (e == cudaSuccess)
        e = awq::launch_act_stats(X, T, K, ldx, reinterpret_cast<unsigned long long*>(abs_sum_q24),
                                  d->status, d->num_sms, st);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

awq_status awq_act_mean(const int64_t* abs_sum_q24, int64_t n_tokens, int64_t K, double* mean_abs,
                        awq_stream_t stream) {
    const CallRange range("awq_act_mean");
    if (n_tokens <= 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "act_mean: n_tokens must be > 0");
    if (K > 0 && (!abs_sum_q24 || !mean_abs)) return fail(AWQ_ERR_INVALID_ARG, "act_mean: null pointer");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaError_t e = awq::launch_act_mean(abs_sum_q24, n_tokens, K, mean_abs, (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

size_t awq_candidate_scales_workspace_size(int64_t K, int n_alpha) {
    if (K <= 0 || n_alpha <= 0) return 0;
    return align256((size_t)n_alpha * K * 8) + align256((size_t)n_alpha * awq::cand_blocks(K) * 16);
}

awq_status awq_candidate_scales(const double* mean_abs, int64_t K, const double* alphas, int n_alpha,
                                float* s_alpha, void* workspace, size_t ws_bytes,
                                awq_stream_t stream) {
    const CallRange range("awq_candidate_scales");
    if (K <= 0 || n_alpha < 1 || n_alpha > AWQ_MAX_ALPHAS)
        return fail(AWQ_ERR_INVALID_ARG, "candidate_scales: bad K or n_alpha");
    if (!mean_abs || !alphas || !s_alpha) return fail(AWQ_ERR_INVALID_ARG, "candidate_scales: null pointer");
    const size_t need = awq_candidate_scales_workspace_size(K, n_alpha);
    if (!workspace || ws_bytes < need || !aligned16(workspace))
        return fail(AWQ_ERR_WORKSPACE, "candidate_scales: workspace missing or too small");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    awq::AlphaList al;
    for (int i = 0; i < n_alpha; ++i) al.a[i] = alphas[i];
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    double* r = reinterpret_cast<double*>(ws);
    double* mm = reinterpret_cast<double*>(ws + align256((size_t)n_alpha * K * 8));
    cudaError_t e = awq::launch_candidate_scales(mean_abs, K, al, n_alpha, s_alpha, nullptr, r, mm,
                                                 (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

size_t awq_search_workspace_size(int64_t N, int64_t K, int64_t T, int n_alpha) {
    if (N <= 0 || K <= 0 || T <= 0 || n_alpha <= 0) return 0;
    return search_ws(N, K, T, n_alpha).total;
}

}  // extern "C"

namespace {

// awq_search_scale and its 3-bit form: levels 0..qmax.
awq_status search_run(DevInfo* d, const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                      const uint16_t* Xcal, int64_t T, int64_t ldx, const float* s_alpha,
                      const float* inv_s, int n_alpha, double* partials, double* mse,
                      int32_t* best_idx, float* s_out, cudaStream_t st, float qmax);

awq_status search_impl(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const uint16_t* Xcal,
                       int64_t T, int64_t ldx, const double* mean_abs, const double* alphas,
                       int n_alpha, int group, float* s_out, double* mse_out, int32_t* best_idx,
                       float* s_alpha_out, void* workspace, size_t ws_bytes, awq_stream_t stream,
                       float qmax) {
    if (N <= 0 || K <= 0 || T <= 0 || n_alpha < 1 || n_alpha > AWQ_MAX_ALPHAS)
        return fail(AWQ_ERR_INVALID_ARG, "search_scale: sizes must be positive, 1 <= n_alpha <= 64");
    if (!W || !Xcal || !mean_abs || !alphas || !s_out || !best_idx)
        return fail(AWQ_ERR_INVALID_ARG, "search_scale: null pointer");
    if (group != AWQ_GROUP || K % AWQ_GROUP || N % 8 || ldw < K || ldx < K || ldw % 8 || ldx % 8)
        return fail(AWQ_ERR_SHAPE, "search_scale: need group 128, K % 128 == 0, N % 8 == 0, ld >= K, ld % 8 == 0");
    if (N > (1LL << 30) || T > (1LL << 30) || K > (1LL << 30))
        return fail(AWQ_ERR_SHAPE, "search_scale: size too large");
    if (!aligned16(W) || !aligned16(Xcal) || !aligned16(s_out) ||
        (s_alpha_out && !aligned16(s_alpha_out)))
        return fail(AWQ_ERR_ALIGN, "search_scale: W, Xcal, s_out must be 16-byte aligned");
    const SearchWs lay = search_ws(N, K, T, n_alpha);
    if (!workspace || ws_bytes < lay.total || !aligned16(workspace))
        return fail(AWQ_ERR_WORKSPACE, "search_scale: workspace missing or too small");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* s_alpha = s_alpha_out ? s_alpha_out : reinterpret_cast<float*>(ws + lay.s_alpha);
    float* inv_s = reinterpret_cast<float*>(ws + lay.inv_s);
    double* partials = reinterpret_cast<double*>(ws + lay.partials);
    double* mse = mse_out ? mse_out : reinterpret_cast<double*>(ws + lay.mse);

    awq::AlphaList al;
    for (int i = 0; i < n_alpha; ++i) al.a[i] = alphas[i];
    cudaError_t e = awq::launch_candidate_scales(mean_abs, K, al, n_alpha, s_alpha, inv_s,
                                                 reinterpret_cast<double*>(ws + lay.r),
                                                 reinterpret_cast<double*>(ws + lay.mm), st);
    if (e != cudaSuccess) return cuda_fail(e);
    return search_run(d, W, N, K, ldw, Xcal, T, ldx, s_alpha, inv_s, n_alpha, partials, mse,
                      best_idx, s_out, st, qmax);
}

// The tensor-core search and the final reduction on candidate scales already
// in place (s_alpha and inv_s, [n_alpha][K] fp32); arguments checked.
awq_status search_run(DevInfo* d, const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                      const uint16_t* Xcal, int64_t T, int64_t ldx, const float* s_alpha,
                      const float* inv_s, int n_alpha, double* partials, double* mse,
                      int32_t* best_idx, float* s_out, cudaStream_t st, float qmax) {
    CUtensorMap map;
    awq_status s = make_act_map(&map, Xcal, T, K, ldx);
    if (s) return s;
    awq::TcParams p = {};
    p.N = (int)N;
    p.K = (int)K;
    p.G = (int)(K / AWQ_GROUP);
    p.rows_tok = (int)T;
    p.n_tiles = (int)((N + awq::kTcRows - 1) / awq::kTcRows);
    p.t_tiles = (int)((T + awq::kSearchTokensPerItem - 1) / awq::kSearchTokensPerItem);
    p.n_alpha = n_alpha;
    p.n_items = p.n_tiles * p.t_tiles * n_alpha;
    p.W = W;
    p.ldw = ldw;
    p.s_alpha = s_alpha;
    p.inv_s_alpha = inv_s;
    p.partials = partials;
    p.status = d->status;
    p.qmax = qmax;
    cudaError_t e = awq::launch_tc_search(map, p, d->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = awq::launch_search_finalize(partials, n_alpha, (int64_t)p.n_tiles * p.t_tiles * 4, T, N, K,
                                    s_alpha, mse, best_idx, s_out, st);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

awq_status awq_search_scale(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                            const uint16_t* Xcal, int64_t T, int64_t ldx, const double* mean_abs,
                            const double* alphas, int n_alpha, int group, float* s_out,
                            double* mse_out, int32_t* best_idx, float* s_alpha_out,
                            void* workspace, size_t ws_bytes, awq_stream_t stream) {
    const CallRange range("awq_search_scale");
    return search_impl(W, N, K, ldw, Xcal, T, ldx, mean_abs, alphas, n_alpha, group, s_out,
                       mse_out, best_idx, s_alpha_out, workspace, ws_bytes, stream, 15.0f);
}

size_t awq_search_mse_workspace_size(int64_t N, int64_t K, int64_t T, int n_alpha) {
    if (N <= 0 || K <= 0 || T <= 0 || n_alpha <= 0) return 0;
    return search_ws(N, K, T, n_alpha).total;
}

awq_status awq_search_mse(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                          const uint16_t* Xcal, int64_t T, int64_t ldx, const float* s_alpha,
                          int n_alpha, int group, float* s_out, double* mse_out,
                          int32_t* best_idx, void* workspace, size_t ws_bytes,
                          awq_stream_t stream) {
    const CallRange range("awq_search_mse");
    if (N <= 0 || K <= 0 || T <= 0 || n_alpha < 1 || n_alpha > AWQ_MAX_ALPHAS)
        return fail(AWQ_ERR_INVALID_ARG, "search_mse: sizes must be positive, 1 <= n_alpha <= 64");
    if (!W || !Xcal || !s_alpha || !s_out || !best_idx)
        return fail(AWQ_ERR_INVALID_ARG, "search_mse: null pointer");
    if (group != AWQ_GROUP || K % AWQ_GROUP || N % 8 || ldw < K || ldx < K || ldw % 8 || ldx % 8)
        return fail(AWQ_ERR_SHAPE, "search_mse: need group 128, K % 128 == 0, N % 8 == 0, ld >= K, ld % 8 == 0");
    if (N > (1LL << 30) || T > (1LL << 30) || K > (1LL << 30))
        return fail(AWQ_ERR_SHAPE, "search_mse: size too large");
    if (!aligned16(W) || !aligned16(Xcal) || !aligned16(s_out) || !aligned16(s_alpha))
        return fail(AWQ_ERR_ALIGN, "search_mse: W, Xcal, s_alpha, s_out must be 16-byte aligned");
    const SearchWs lay = search_ws(N, K, T, n_alpha);
    if (!workspace || ws_bytes < lay.total || !aligned16(workspace))
        return fail(AWQ_ERR_WORKSPACE, "search_mse: workspace missing or too small");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* inv_s = reinterpret_cast<float*>(ws + lay.inv_s);
    double* partials = reinterpret_cast<double*>(ws + lay.partials);
    double* mse = mse_out ? mse_out : reinterpret_cast<double*>(ws + lay.mse);
    cudaError_t e = awq::launch_reciprocals(s_alpha, (int64_t)n_alpha * K, inv_s, d->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return search_run(d, W, N, K, ldw, Xcal, T, ldx, s_alpha, inv_s, n_alpha, partials, mse,
                      best_idx, s_out, st, 15.0f);
}

awq_status awq_search_scale_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                 const uint16_t* Xcal, int64_t T, int64_t ldx,
                                 const double* mean_abs, const double* alphas, int n_alpha,
                                 int group, float* s_out, double* mse_out, int32_t* best_idx,
                                 float* s_alpha_out, void* workspace, size_t ws_bytes,
                                 awq_stream_t stream) {
    const CallRange range("awq_search_scale_int3");
    return search_impl(W, N, K, ldw, Xcal, T, ldx, mean_abs, alphas, n_alpha, group, s_out,
                       mse_out, best_idx, s_alpha_out, workspace, ws_bytes, stream, 7.0f);
}

// Tokens of the transposed copy: T rounded up to a whole 64-token TMA box.
static int64_t gram_t_pad(int64_t T) { return (T + 63) / 64 * 64; }

size_t awq_gram_workspace_size(int64_t T, int64_t K) {
    if (T <= 0 || K <= 0) return 0;
    return align256((size_t)K * (size_t)gram_t_pad(T) * 2);
}

awq_status awq_gram(const uint16_t* Xcal, int64_t T, int64_t K, int64_t ldx, uint16_t* G,
                    void* workspace, size_t ws_bytes, awq_stream_t stream) {
    const CallRange range("awq_gram");
    if (T <= 0 || K <= 0) return fail(AWQ_ERR_INVALID_ARG, "gram: sizes must be positive");
    if (!Xcal || !G) return fail(AWQ_ERR_INVALID_ARG, "gram: null pointer");
    if (K % AWQ_GROUP || ldx < K || ldx % 8)
        return fail(AWQ_ERR_SHAPE, "gram: need K % 128 == 0, ldx >= K, ldx % 8 == 0");
    if (T > (1LL << 30) || K > (1LL << 22))
        return fail(AWQ_ERR_SHAPE, "gram: size too large");
    if (!aligned16(Xcal) || !aligned16(G))
        return fail(AWQ_ERR_ALIGN, "gram: Xcal and G must be 16-byte aligned");
    const size_t need = awq_gram_workspace_size(T, K);
    if (!workspace || ws_bytes < need || !aligned16(workspace))
        return fail(AWQ_ERR_WORKSPACE, "gram: workspace missing or too small");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t T_pad = gram_t_pad(T);
    uint16_t* Xt = static_cast<uint16_t*>(workspace);
    cudaError_t e = awq::launch_transpose_x(Xcal, T, K, ldx, Xt, T_pad, st);
    if (e != cudaSuccess) return cuda_fail(e);
    // X^T [K][T_pad]: B boxes of 64 tokens x 256 rows, A boxes of 64 x 128
    CUtensorMap mapB, mapA;
    s = make_act_map(&mapB, Xt, K, T_pad, T_pad);
    if (s) return s;
    s = make_map_rows(&mapA, Xt, K, T_pad, T_pad, awq::kTcRows);
    if (s) return s;
    awq::TcParams p = {};
    p.N = (int)K;
    p.K = (int)T_pad;
    p.G = (int)((T_pad + AWQ_GROUP - 1) / AWQ_GROUP);
    p.rows_tok = (int)K;
    p.n_tiles = (int)(K / awq::kTcRows);
    p.t_tiles = (int)((K + awq::kSearchTokensPerItem - 1) / awq::kSearchTokensPerItem);
    p.n_items = p.n_tiles * p.t_tiles;
    p.gout = G;
    p.inv_t = (float)(1.0 / (double)T);
    p.status = d->status;
    e = awq::launch_tc_xtx(mapB, mapA, p, d->num_sms, st);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

size_t awq_search_gram_workspace_size(int64_t N, int64_t K, int n_alpha) {
    if (N <= 0 || K <= 0 || n_alpha <= 0) return 0;
    return search_ws(N, K, K, n_alpha).total + gram_exp_bytes(current_num_sms());
}

}  // extern "C"

namespace {

awq_status search_gram_impl(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const uint16_t* G,
                            const double* mean_abs, const double* alphas, int n_alpha, int group,
                            float* s_out, double* mse_out, int32_t* best_idx, float* s_alpha_out,
                            void* workspace, size_t ws_bytes, awq_stream_t stream, float qmax) {
    if (N <= 0 || K <= 0 || n_alpha < 1 || n_alpha > AWQ_MAX_ALPHAS)
        return fail(AWQ_ERR_INVALID_ARG, "search_scale_gram: sizes must be positive, 1 <= n_alpha <= 64");
    if (!W || !G || !mean_abs || !alphas || !s_out || !best_idx)
        return fail(AWQ_ERR_INVALID_ARG, "search_scale_gram: null pointer");
    if (group != AWQ_GROUP || K % AWQ_GROUP || N % 8 || ldw < K || ldw % 8)
        return fail(AWQ_ERR_SHAPE, "search_scale_gram: need group 128, K % 128 == 0, N % 8 == 0, ldw >= K, ldw % 8 == 0");
    if (N > (1LL << 30) || K > (1LL << 22))
        return fail(AWQ_ERR_SHAPE, "search_scale_gram: size too large");
    if (!aligned16(W) || !aligned16(G) || !aligned16(s_out) ||
        (s_alpha_out && !aligned16(s_alpha_out)))
        return fail(AWQ_ERR_ALIGN, "search_scale_gram: W, G, s_out must be 16-byte aligned");
    const SearchWs lay = search_ws(N, K, K, n_alpha);
    if (!workspace || ws_bytes < lay.total || !aligned16(workspace))
        return fail(AWQ_ERR_WORKSPACE, "search_scale_gram: workspace missing or too small");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    // (the residual hand-over buffers scale with the device's SM count)
    if (ws_bytes < lay.total + gram_exp_bytes(d->num_sms))
        return fail(AWQ_ERR_WORKSPACE, "search_scale_gram: workspace missing or too small");
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* s_alpha = s_alpha_out ? s_alpha_out : reinterpret_cast<float*>(ws + lay.s_alpha);
    float* inv_s = reinterpret_cast<float*>(ws + lay.inv_s);
    double* partials = reinterpret_cast<double*>(ws + lay.partials);
    double* mse = mse_out ? mse_out : reinterpret_cast<double*>(ws + lay.mse);
    awq::AlphaList al;
    for (int i = 0; i < n_alpha; ++i) al.a[i] = alphas[i];
    cudaError_t e = awq::launch_candidate_scales(mean_abs, K, al, n_alpha, s_alpha, inv_s,
                                                 reinterpret_cast<double*>(ws + lay.r),
                                                 reinterpret_cast<double*>(ws + lay.mm), st);
    if (e != cudaSuccess) return cuda_fail(e);
    CUtensorMap map;
    s = make_act_map(&map, G, K, K, K);
    if (s) return s;
    awq::TcParams p = {};
    p.N = (int)N;
    p.K = (int)K;
    p.G = (int)(K / AWQ_GROUP);
    p.rows_tok = (int)K;
    p.n_tiles = (int)((N + awq::kTcRows - 1) / awq::kTcRows);
    p.t_tiles = (int)((K + awq::kSearchTokensPerItem - 1) / awq::kSearchTokensPerItem);
    p.n_alpha = n_alpha;
    p.n_items = p.n_tiles * p.t_tiles * n_alpha;
    p.W = W;
    p.ldw = ldw;
    p.s_alpha = s_alpha;
    p.inv_s_alpha = inv_s;
    p.partials = partials;
    p.status = d->status;
    p.qmax = qmax;
    p.e_exp = reinterpret_cast<uint16_t*>(ws + lay.total);
    e = awq::launch_tc_gram_search(map, p, d->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e);
    // G already carries the 1/T of the mean: divide the sums by N only
    e = awq::launch_search_finalize(partials, n_alpha, (int64_t)p.n_tiles * p.t_tiles * 4, 1, N, K,
                                    s_alpha, mse, best_idx, s_out, st);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

awq_status awq_search_scale_gram(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                 const uint16_t* G, const double* mean_abs, const double* alphas,
                                 int n_alpha, int group, float* s_out, double* mse_out,
                                 int32_t* best_idx, float* s_alpha_out, void* workspace,
                                 size_t ws_bytes, awq_stream_t stream) {
    const CallRange range("awq_search_scale_gram");
    return search_gram_impl(W, N, K, ldw, G, mean_abs, alphas, n_alpha, group, s_out, mse_out,
                            best_idx, s_alpha_out, workspace, ws_bytes, stream, 15.0f);
}

awq_status awq_search_scale_gram_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                      const uint16_t* G, const double* mean_abs,
                                      const double* alphas, int n_alpha, int group, float* s_out,
                                      double* mse_out, int32_t* best_idx, float* s_alpha_out,
                                      void* workspace, size_t ws_bytes, awq_stream_t stream) {
    const CallRange range("awq_search_scale_gram_int3");
    return search_gram_impl(W, N, K, ldw, G, mean_abs, alphas, n_alpha, group, s_out, mse_out,
                            best_idx, s_alpha_out, workspace, ws_bytes, stream, 7.0f);
}

awq_status awq_pack_int4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                         int group, uint32_t* qweight, uint16_t* scales, uint16_t* zeros,
                         awq_stream_t stream) {
    const CallRange range("awq_pack_int4");
    if (N < 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "pack_int4: negative size");
    if ((N > 0 && K > 0) && (!W || !qweight || !scales || !zeros))
        return fail(AWQ_ERR_INVALID_ARG, "pack_int4: null pointer");
    if (group != AWQ_GROUP || K % AWQ_GROUP || ldw < K || ldw % 8)
        return fail(AWQ_ERR_SHAPE, "pack_int4: need group 128, K % 128 == 0, ldw >= K, ldw % 8 == 0");
    if ((W && !aligned16(W)) || (qweight && !aligned16(qweight)) || (s && !aligned16(s)) ||
        (reinterpret_cast<uintptr_t>(scales) & 1u) || (reinterpret_cast<uintptr_t>(zeros) & 1u))
        return fail(AWQ_ERR_ALIGN, "pack_int4: W, qweight, s must be 16-byte aligned");
    DevInfo* d = nullptr;
    awq_status st_ = device_info(&d);
    if (st_) return st_;
    cudaError_t e = awq::launch_pack_int4(W, N, K, ldw, s, qweight, scales, zeros, d->status,
                                          d->num_sms, (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

awq_status w3a16_gemm(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                      const uint32_t* planes, const uint16_t* scales, const uint16_t* zeros,
                      int64_t N, int group, uint16_t* Y, int64_t ldy, awq_stream_t stream) {
    const CallRange range("w3a16_gemm");
    if (M < 0 || N < 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "w3a16_gemm: negative size");
    if (M == 0 || N == 0) return AWQ_OK;
    if (!X || !planes || !scales || !zeros || !Y)
        return fail(AWQ_ERR_INVALID_ARG, "w3a16_gemm: null pointer");
    if (group != AWQ_GROUP || K <= 0 || K % AWQ_GROUP || N % 8 || ldx < K || ldx % 8 || ldy < N)
        return fail(AWQ_ERR_SHAPE, "w3a16_gemm: need group 128, K % 128 == 0, N % 8 == 0, ldx >= K, ldx % 8 == 0, ldy >= N");
    if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30))
        return fail(AWQ_ERR_SHAPE, "w3a16_gemm: size too large");
    if (!aligned16(X) || (reinterpret_cast<uintptr_t>(planes) & 3u) ||
        (M > 16 && !aligned16(planes)) || (reinterpret_cast<uintptr_t>(Y) & 1u) ||
        (reinterpret_cast<uintptr_t>(scales) & 1u) || (reinterpret_cast<uintptr_t>(zeros) & 1u))
        return fail(AWQ_ERR_ALIGN, "w3a16_gemm: X must be 16-byte aligned, planes 4-byte (16-byte for M > 16)");
    DevInfo* d = nullptr;
    awq_status st_ = device_info(&d);
    if (st_) return st_;
    cudaError_t e;
    if (M <= 16) {
        e = awq::launch_gemv_w3a16(X, ldx, (int)M, planes, scales, zeros, N, K, Y, ldy,
                                   d->num_sms, (cudaStream_t)stream);
    } else {
        // prefill: the tcgen05 GEMM with a producer that rebuilds fp16 levels
        // from the planes (no split of K, so no workspace)
        CUtensorMap map;
        awq_status s = make_act_map(&map, X, M, K, ldx);
        if (s) return s;
        awq::TcParams p = {};
        p.N = (int)N;
        p.K = (int)K;
        p.G = (int)(K / AWQ_GROUP);
        p.rows_tok = (int)M;
        p.n_tiles = (int)((N + awq::kTcRows - 1) / awq::kTcRows);
        p.t_tiles = (int)((M + awq::kGemmTokensPerItem - 1) / awq::kGemmTokensPerItem);
        p.k_splits = 1;
        p.n_items = p.n_tiles * p.t_tiles;
        p.planes = planes;
        p.scales = scales;
        p.zeros = zeros;
        p.Y = Y;
        p.ldy = ldy;
        p.status = d->status;
        p.early_w = g_early_weights.load(std::memory_order_relaxed);
        e = awq::launch_tc_gemm3(map, p, d->num_sms, (cudaStream_t)stream);
    }
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

awq_status awq_pack_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                         int group, uint32_t* planes, uint16_t* scales, uint16_t* zeros,
                         awq_stream_t stream) {
    const CallRange range("awq_pack_int3");
    if (N < 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "pack_int3: negative size");
    if ((N > 0 && K > 0) && (!W || !planes || !scales || !zeros))
        return fail(AWQ_ERR_INVALID_ARG, "pack_int3: null pointer");
    if (group != AWQ_GROUP || K % AWQ_GROUP || ldw < K || ldw % 8)
        return fail(AWQ_ERR_SHAPE, "pack_int3: need group 128, K % 128 == 0, ldw >= K, ldw % 8 == 0");
    if ((W && !aligned16(W)) || (s && !aligned16(s)) ||
        (reinterpret_cast<uintptr_t>(planes) & 3u) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
        (reinterpret_cast<uintptr_t>(zeros) & 1u))
        return fail(AWQ_ERR_ALIGN, "pack_int3: W, s must be 16-byte aligned, planes 4-byte");
    DevInfo* d = nullptr;
    awq_status st_ = device_info(&d);
    if (st_) return st_;
    cudaError_t e = awq::launch_pack_int3(W, N, K, ldw, s, planes, scales, zeros, d->status,
                                          d->num_sms, (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

// Work split of the tensor-core GEMM.  The modelled time is waves x
// (groups per item) x (one group of one 128 x 256 tile, about 1 us on B300)
// plus the partials' extra traffic (written and read once, fp32, at about
// 5 TB/s).  Two ways to fill the grid beside plain whole tiles:
//  - K splits: every tile's K range in k_splits equal parts (fp32 partials
//    laid out like Y); pays for under-filled grids with long K;
//  - stream-K tail: whole waves of tiles, then the K range of the remaining
//    tiles (fewer than the SMs) cut into equal shares, one per SM (fp32
//    partial tiles, two slots per SM), so the last wave is not mostly idle.
// A split must win clearly (3%) over the plainer schedule.
struct GemmSched {
    int k_splits = 1;
    int sk_full = 0, sk_tiles = 0;     // stream-K tail when sk_tiles > 0
};

GemmSched gemm_schedule(int64_t M, int64_t N, int64_t K, int num_sms) {
    GemmSched sc;
    if (M <= 16 || num_sms <= 0) return sc;
    const int64_t G = K / AWQ_GROUP;
    const int64_t tiles = ((N + awq::kTcRows - 1) / awq::kTcRows) *
                          ((M + awq::kGemmTokensPerItem - 1) / awq::kGemmTokensPerItem);
    double best_t = 1e300;
    for (int ks = 1; ks <= 8; ++ks) {
        if (G / ks < 4) break;
        const int64_t waves = (tiles * ks + num_sms - 1) / num_sms;
        const double t = (double)waves * ((double)G / ks) * 1e-6 +
                         (ks > 1 ? 2.0 * ks * (double)M * (double)N * 4.0 / 5e12 : 0.0);
        if (t < best_t * 0.97) {
            best_t = t;
            sc.k_splits = ks;
        }
    }
    const int64_t R = tiles % num_sms;
    if (R > 0 && G >= 4 && num_sms <= 256) {      // (the fixup lists <= 512 slots a tile)
        const double tile_bytes = (double)awq::kTcRows * awq::kTcTokens * 4.0;
        const double t = (double)(tiles / num_sms) * (double)G * 1e-6 +
                         std::ceil((double)(R * G) / num_sms) * 1e-6 +
                         2.0 * (double)(num_sms + R) * tile_bytes / 5e12 + 3e-6;
        if (t < best_t * 0.97) {
            sc.k_splits = 1;
            sc.sk_full = (int)(tiles - R);
            sc.sk_tiles = (int)R;
        }
    }
    return sc;
}

// Workspace bytes of a schedule (after the scaled-X pre-pass's share).
size_t sched_ws_bytes(const GemmSched& sc, int64_t M, int64_t N, int num_sms) {
    if (sc.sk_tiles > 0)
        return (size_t)2 * (size_t)num_sms * awq::kTcRows * awq::kTcTokens * sizeof(float);
    return sc.k_splits > 1 ? (size_t)sc.k_splits * (size_t)M * (size_t)N * sizeof(float) : 0;
}

int current_num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

extern "C" {

size_t w4a16_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (M <= 16 || N <= 0 || K <= 0 || K % AWQ_GROUP) return 0;
    const int sms = current_num_sms();
    return sched_ws_bytes(gemm_schedule(M, N, K, sms), M, N, sms);
}

}  // extern "C"

namespace {

// Bytes the fused-scaling pre-pass needs in front of the GEMM's own
// workspace (M > 16 only).
size_t scaled_x_bytes(int64_t M, int64_t K) {
    return M > 16 ? align256((size_t)M * (size_t)K * 2) : 0;
}

// w4a16_gemm and w4a16_gemm_scaled: inv_s null for the plain call.
awq_status gemm_impl(const char* name, const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                     const float* inv_s, const uint32_t* qweight, const uint16_t* scales,
                     const uint16_t* zeros, int64_t N, int group, uint16_t* Y, int64_t ldy,
                     void* workspace, size_t ws_bytes, awq_stream_t stream) {
    if (M < 0 || N < 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "w4a16_gemm: negative size");
    if (M == 0 || N == 0) return AWQ_OK;
    if (!X || !qweight || !scales || !zeros || !Y)
        return fail(AWQ_ERR_INVALID_ARG, "w4a16_gemm: null pointer");
    if (group != AWQ_GROUP || K <= 0 || K % AWQ_GROUP || N % 8 || ldx < K || ldx % 8 || ldy < N)
        return fail(AWQ_ERR_SHAPE, "w4a16_gemm: need group 128, K % 128 == 0, N % 8 == 0, ldx >= K, ldx % 8 == 0, ldy >= N");
    if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30))
        return fail(AWQ_ERR_SHAPE, "w4a16_gemm: size too large");
    if (!aligned16(X) || !aligned16(qweight) || (reinterpret_cast<uintptr_t>(Y) & 1u) ||
        (reinterpret_cast<uintptr_t>(scales) & 1u) || (reinterpret_cast<uintptr_t>(zeros) & 1u) ||
        (inv_s && !aligned16(inv_s)))
        return fail(AWQ_ERR_ALIGN, "w4a16_gemm: X, qweight (and inv_s) must be 16-byte aligned");
    (void)name;
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (M <= 16) {
        CUtensorMap map;
        s = make_qweight_map(&map, qweight, N, K);
        if (s) return s;
        awq::GemvParams p = {X, ldx, (int)M, qweight, scales, zeros, N, K, (int)(K / AWQ_GROUP),
                             Y, ldy, d->status, g_early_weights.load(std::memory_order_relaxed),
                             inv_s};
        e = awq::launch_gemv(map, p, d->num_sms, st);
    } else {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        const size_t xs_bytes = inv_s ? scaled_x_bytes(M, K) : 0;
        const GemmSched sc = gemm_schedule(M, N, K, d->num_sms);
        const int k_splits = sc.k_splits;
        const size_t part_bytes = sched_ws_bytes(sc, M, N, d->num_sms);
        if ((xs_bytes + part_bytes) > 0 &&
            (!workspace || ws_bytes < xs_bytes + part_bytes || !aligned16(workspace)))
            return fail(AWQ_ERR_WORKSPACE, "w4a16_gemm: workspace missing or too small "
                                           "(see w4a16_gemm_workspace_size)");
        const uint16_t* Xa = X;
        int64_t lda = ldx;
        if (inv_s) {   // pre-pass: fp16(X * inv_s) into the workspace
            uint16_t* Xs = reinterpret_cast<uint16_t*>(ws);
            e = awq::launch_scale_x(X, M, K, ldx, inv_s, Xs, d->num_sms, st);
            if (e != cudaSuccess) return cuda_fail(e);
            Xa = Xs;
            lda = K;
        }
        CUtensorMap map, mapW;
        s = make_act_map(&map, Xa, M, K, lda);
        if (s) return s;
        s = make_qweight_map(&mapW, qweight, N, K, kQwGemm);
        if (s) return s;
        awq::TcParams p = {};
        p.N = (int)N;
        p.K = (int)K;
        p.G = (int)(K / AWQ_GROUP);
        p.rows_tok = (int)M;
        p.n_tiles = (int)((N + awq::kTcRows - 1) / awq::kTcRows);
        p.t_tiles = (int)((M + awq::kGemmTokensPerItem - 1) / awq::kGemmTokensPerItem);
        p.k_splits = k_splits;
        p.n_items = p.n_tiles * p.t_tiles * k_splits;
        if (sc.sk_tiles > 0) {
            p.sk_full = sc.sk_full;
            p.sk_tiles = sc.sk_tiles;
            p.sk_ctas = d->num_sms;
            p.n_items = sc.sk_full + d->num_sms;      // launches sk_ctas CTAs
            p.ws_sk = reinterpret_cast<float*>(ws + xs_bytes);
        }
        p.qw = qweight;
        p.scales = scales;
        p.zeros = zeros;
        p.Y = Y;
        p.ldy = ldy;
        p.status = d->status;
        // after the scaling pre-pass (which writes only Xs) the weights may
        // be read early; otherwise only when the caller allows it
        p.early_w = inv_s ? 1 : g_early_weights.load(std::memory_order_relaxed);
        if (k_splits > 1) p.ws_partial = reinterpret_cast<float*>(ws + xs_bytes);
        e = awq::launch_tc_gemm(map, mapW, p, d->num_sms, st);
        if (e == cudaSuccess && k_splits > 1)
            e = awq::launch_splitk_reduce(p.ws_partial, k_splits, M, N, Y, ldy, d->num_sms, st);
        if (e == cudaSuccess && p.sk_tiles > 0) e = awq::launch_sk_fixup(p, st);
    }
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

awq_status w4a16_gemm(const uint16_t* X, int64_t M, int64_t K, int64_t ldx, const uint32_t* qweight,
                      const uint16_t* scales, const uint16_t* zeros, int64_t N, int group,
                      uint16_t* Y, int64_t ldy, void* workspace, size_t ws_bytes,
                      awq_stream_t stream) {
    const CallRange range("w4a16_gemm");
    return gemm_impl("w4a16_gemm", X, M, K, ldx, nullptr, qweight, scales, zeros, N, group, Y,
                     ldy, workspace, ws_bytes, stream);
}

size_t awq_repack_int4_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % AWQ_GROUP) return 0;
    return (size_t)((N + 15) / 16) * (size_t)(K / AWQ_GROUP) * (size_t)awq::kTileBytes;
}

awq_status awq_repack_int4(const uint32_t* qweight, const uint16_t* scales, const uint16_t* zeros,
                           int64_t N, int64_t K, int group, void* tiles, size_t tiles_bytes,
                           awq_stream_t stream) {
    const CallRange range("awq_repack_int4");
    if (N < 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "repack_int4: negative size");
    if (N == 0 || K == 0) return AWQ_OK;
    if (!qweight || !scales || !zeros || !tiles)
        return fail(AWQ_ERR_INVALID_ARG, "repack_int4: null pointer");
    if (group != AWQ_GROUP || K % AWQ_GROUP || N > (1LL << 30) || K > (1LL << 30))
        return fail(AWQ_ERR_SHAPE, "repack_int4: need group 128, K % 128 == 0");
    if (!aligned16(qweight) || !aligned16(tiles) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
        (reinterpret_cast<uintptr_t>(zeros) & 1u))
        return fail(AWQ_ERR_ALIGN, "repack_int4: qweight and tiles must be 16-byte aligned");
    if (tiles_bytes < awq_repack_int4_bytes(N, K))
        return fail(AWQ_ERR_WORKSPACE, "repack_int4: tiles buffer smaller than awq_repack_int4_bytes(N, K)");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaError_t e = awq::launch_repack_int4(qweight, scales, zeros, N, K, tiles, d->num_sms,
                                            (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

awq_status w4a16_gemm_repacked(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                               const float* inv_s, const void* tiles, int64_t N, int group,
                               uint16_t* Y, int64_t ldy, awq_stream_t stream) {
    const CallRange range("w4a16_gemm_repacked");
    if (M < 0 || N < 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "w4a16_gemm_repacked: negative size");
    if (M == 0 || N == 0) return AWQ_OK;
    if (!X || !tiles || !Y) return fail(AWQ_ERR_INVALID_ARG, "w4a16_gemm_repacked: null pointer");
    if (M > 16 || group != AWQ_GROUP || K <= 0 || K % AWQ_GROUP || N % 8 || ldx < K || ldx % 8 ||
        ldy < N)
        return fail(AWQ_ERR_SHAPE, "w4a16_gemm_repacked: need M <= 16, group 128, K % 128 == 0, N % 8 == 0, ldx >= K, ldx % 8 == 0, ldy >= N");
    if (N > (1LL << 30) || K > (1LL << 30))
        return fail(AWQ_ERR_SHAPE, "w4a16_gemm_repacked: size too large");
    if (!aligned16(X) || !aligned16(tiles) || (reinterpret_cast<uintptr_t>(Y) & 1u) ||
        (inv_s && !aligned16(inv_s)))
        return fail(AWQ_ERR_ALIGN, "w4a16_gemm_repacked: X, tiles (and inv_s) must be 16-byte aligned");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    awq::TileParams p = {X, ldx, (int)M, static_cast<const uint8_t*>(tiles), N,
                         (int)(K / AWQ_GROUP), Y, ldy, d->status,
                         g_early_weights.load(std::memory_order_relaxed), inv_s, 4};
    cudaError_t e = awq::launch_gemv_tiles(p, d->num_sms, (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

size_t awq_repack_int3_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % AWQ_GROUP) return 0;
    return (size_t)((N + 15) / 16) * (size_t)(K / AWQ_GROUP) * (size_t)awq::kTile3Bytes;
}

awq_status awq_repack_int3(const uint32_t* planes, const uint16_t* scales, const uint16_t* zeros,
                           int64_t N, int64_t K, int group, void* tiles, size_t tiles_bytes,
                           awq_stream_t stream) {
    const CallRange range("awq_repack_int3");
    if (N < 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "repack_int3: negative size");
    if (N == 0 || K == 0) return AWQ_OK;
    if (!planes || !scales || !zeros || !tiles)
        return fail(AWQ_ERR_INVALID_ARG, "repack_int3: null pointer");
    if (group != AWQ_GROUP || K % AWQ_GROUP || N > (1LL << 30) || K > (1LL << 30))
        return fail(AWQ_ERR_SHAPE, "repack_int3: need group 128, K % 128 == 0");
    if (!aligned16(planes) || !aligned16(tiles) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
        (reinterpret_cast<uintptr_t>(zeros) & 1u))
        return fail(AWQ_ERR_ALIGN, "repack_int3: planes and tiles must be 16-byte aligned");
    if (tiles_bytes < awq_repack_int3_bytes(N, K))
        return fail(AWQ_ERR_WORKSPACE, "repack_int3: tiles buffer smaller than awq_repack_int3_bytes(N, K)");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    cudaError_t e = awq::launch_repack_int3(planes, scales, zeros, N, K, tiles, d->num_sms,
                                            (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

awq_status w3a16_gemm_repacked(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                               const void* tiles, int64_t N, int group, uint16_t* Y, int64_t ldy,
                               awq_stream_t stream) {
    const CallRange range("w3a16_gemm_repacked");
    if (M < 0 || N < 0 || K < 0) return fail(AWQ_ERR_INVALID_ARG, "w3a16_gemm_repacked: negative size");
    if (M == 0 || N == 0) return AWQ_OK;
    if (!X || !tiles || !Y) return fail(AWQ_ERR_INVALID_ARG, "w3a16_gemm_repacked: null pointer");
    if (M > 16 || group != AWQ_GROUP || K <= 0 || K % AWQ_GROUP || N % 8 || ldx < K || ldx % 8 ||
        ldy < N)
        return fail(AWQ_ERR_SHAPE, "w3a16_gemm_repacked: need M <= 16, group 128, K % 128 == 0, N % 8 == 0, ldx >= K, ldx % 8 == 0, ldy >= N");
    if (N > (1LL << 30) || K > (1LL << 30))
        return fail(AWQ_ERR_SHAPE, "w3a16_gemm_repacked: size too large");
    if (!aligned16(X) || !aligned16(tiles) || (reinterpret_cast<uintptr_t>(Y) & 1u))
        return fail(AWQ_ERR_ALIGN, "w3a16_gemm_repacked: X and tiles must be 16-byte aligned");
    DevInfo* d = nullptr;
    awq_status s = device_info(&d);
    if (s) return s;
    awq::TileParams p = {X, ldx, (int)M, static_cast<const uint8_t*>(tiles), N,
                         (int)(K / AWQ_GROUP), Y, ldy, d->status,
                         g_early_weights.load(std::memory_order_relaxed), nullptr, 3};
    cudaError_t e = awq::launch_gemv_tiles(p, d->num_sms, (cudaStream_t)stream);
    return e == cudaSuccess ? AWQ_OK : cuda_fail(e);
}

size_t w4a16_gemm_scaled_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % AWQ_GROUP) return 0;
    return scaled_x_bytes(M, K) + w4a16_gemm_workspace_size(M, N, K);
}

awq_status w4a16_gemm_scaled(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                             const float* inv_s, const uint32_t* qweight, const uint16_t* scales,
                             const uint16_t* zeros, int64_t N, int group, uint16_t* Y, int64_t ldy,
                             void* workspace, size_t ws_bytes, awq_stream_t stream) {
    const CallRange range("w4a16_gemm_scaled");
    if (!inv_s) return fail(AWQ_ERR_INVALID_ARG, "w4a16_gemm_scaled: null inv_s");
    return gemm_impl("w4a16_gemm_scaled", X, M, K, ldx, inv_s, qweight, scales, zeros, N, group,
                     Y, ldy, workspace, ws_bytes, stream);
}

}  // extern "C"
