// Calibration statistics: per-input-channel sum of |x| (the pages' "average
// activation magnitude" of "AWQ: Activation-aware Weight Quantization ...",
// third paragraph; statistics only, seventh paragraph).
//
// Every finite fp16 value is an integer multiple of 2^-24 below 2^16, so
// |x| * 2^24 is an integer below 2^40 and the per-channel sum is accumulated
// exactly in 64-bit integers: any 2^23 - 1 tokens sum to less than 2^63.  Integer addition is associative, so the
// result is bit-identical whatever the order of threads, blocks or atomics.
#include "common.cuh"
#include "kernels.cuh"

namespace awq {
namespace {

constexpr int kStatCols = 256;   // columns per block (32 lanes x 8)
constexpr int kStatRowLanes = 8; // warps per block, each striding rows

__device__ __forceinline__ uint64_t abs_q24(uint32_t h, bool& bad) {
    uint32_t e = (h >> 10) & 31u, f = h & 1023u;
    if (e == 31u) {
        bad = true;
        return 0;
    }
    return e ? (uint64_t)(1024u + f) << (e - 1u) : (uint64_t)f;
}

__global__ void __launch_bounds__(kStatCols)
    act_stats_kernel(const uint16_t* __restrict__ X, int64_t T, int64_t K, int64_t ldx,
                     int64_t rows_per_block, unsigned long long* __restrict__ abs_sum,
                     unsigned* status) {
    __shared__ unsigned long long red[kStatRowLanes][kStatCols + 1];
    const int lx = threadIdx.x & 31, ly = threadIdx.x >> 5;
    const int64_t c0 = (int64_t)blockIdx.x * kStatCols + lx * 8;
    const int64_t r0 = (int64_t)blockIdx.y * rows_per_block;
    const int64_t r1 = min(T, r0 + rows_per_block);
    uint64_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    bool bad = false;
    if (c0 < K) {
        int64_t r = r0 + ly;
        // two rows in flight per thread
        for (; r + kStatRowLanes < r1; r += 2 * kStatRowLanes) {
            uint4 v0 = __ldg(reinterpret_cast<const uint4*>(X + r * ldx + c0));
            uint4 v1 = __ldg(reinterpret_cast<const uint4*>(X + (r + kStatRowLanes) * ldx + c0));
            uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc[(2 * i) & 7] += abs_q24(w[i] & 0xFFFFu, bad);
                acc[(2 * i + 1) & 7] += abs_q24(w[i] >> 16, bad);
            }
        }
        if (r < r1) {
            uint4 v0 = __ldg(reinterpret_cast<const uint4*>(X + r * ldx + c0));
            uint32_t w[4] = {v0.x, v0.y, v0.z, v0.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] += abs_q24(w[i] & 0xFFFFu, bad);
                acc[2 * i + 1] += abs_q24(w[i] >> 16, bad);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) red[ly][lx * 8 + j] = acc[j];
    __syncthreads();
    const int64_t col = (int64_t)blockIdx.x * kStatCols + threadIdx.x;
    if (col < K) {
        unsigned long long s = 0;
#pragma unroll
        for (int y = 0; y < kStatRowLanes; ++y) s += red[y][threadIdx.x];
        // the running total must stay below 2^63 (a non-negative int64);
        // a call adds less than 2^63 (fewer than 2^23 tokens, each term
        // below 2^40), so reaching bit 63 or wrapping is detected here
        if (s) {
            const unsigned long long old = atomicAdd(abs_sum + col, s);
            if (old + s < old || ((old + s) >> 63)) set_status(status, kStatusOverflow);
        }
    }
    if (bad) set_status(status, kStatusNonFinite);
}

__global__ void act_mean_kernel(const int64_t* __restrict__ abs_sum, int64_t n_tokens, int64_t K,
                                double* __restrict__ mean) {
    int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < K) mean[k] = ((double)abs_sum[k] / 16777216.0) / (double)n_tokens;
}

// Diagnostic: one warp waits, with the kernels' bounded wait and a short
// limit, for phase 0 of an mbarrier that nothing arrives on.  The wait runs
// out, records the timeout status and the kernel returns.
__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns, unsigned* status) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(&bar, 0, &abort, status, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, unsigned* status,
                                         cudaStream_t st) {
    wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, status);
    return cudaGetLastError();
}

cudaError_t launch_act_stats(const uint16_t* X, int64_t T, int64_t K, int64_t ldx,
                             unsigned long long* abs_sum, unsigned* status, int num_sms,
                             cudaStream_t st) {
    if (T == 0 || K == 0) return cudaSuccess;
    const int64_t col_blocks = (K + kStatCols - 1) / kStatCols;
    // aim for about four blocks per SM, each covering at least 64 rows
    int64_t want_row_blocks = (4LL * num_sms + col_blocks - 1) / col_blocks;
    int64_t rows = (T + want_row_blocks - 1) / want_row_blocks;
    rows = ((rows < 64 ? 64 : rows) + 15) / 16 * 16;
    int64_t row_blocks = (T + rows - 1) / rows;
    if (row_blocks > 65535) {
        row_blocks = 65535;
        rows = ((T + row_blocks - 1) / row_blocks + 15) / 16 * 16;
        row_blocks = (T + rows - 1) / rows;
    }
    dim3 grid((unsigned)col_blocks, (unsigned)row_blocks);
    act_stats_kernel<<<grid, kStatCols, 0, st>>>(X, T, K, ldx, rows, abs_sum, status);
    return cudaGetLastError();
}

cudaError_t launch_act_mean(const int64_t* abs_sum, int64_t n_tokens, int64_t K, double* mean,
                            cudaStream_t st) {
    if (K == 0) return cudaSuccess;
    act_mean_kernel<<<(unsigned)((K + 255) / 256), 256, 0, st>>>(abs_sum, n_tokens, K, mean);
    return cudaGetLastError();
}

}  // namespace awq
