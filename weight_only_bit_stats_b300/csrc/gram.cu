// Transposed copy of the calibration activations for the Gram-matrix route of
// the alpha search: X [T][K] -> X^T [K][T_pad], columns T..T_pad-1 zero.
// Both operands of G = X^T X then have the contraction index (the token) as
// their contiguous dimension, which is what the K-major tensor-core tiles of
// tc.cu load.  Memory-bound; 64 x 64 tiles through shared memory so that
// reads and writes are both row-contiguous.
#include "common.cuh"
#include "kernels.cuh"

namespace awq {
namespace {

constexpr int kTr = 64;

__global__ void __launch_bounds__(256)
    transpose_x_kernel(const uint16_t* __restrict__ X, int64_t T, int64_t K, int64_t ldx,
                       uint16_t* __restrict__ Xt, int64_t T_pad) {
    __shared__ uint16_t tile[kTr][kTr + 2];
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;     // 64 x 4 threads
    const int64_t t0 = (int64_t)blockIdx.x * kTr, k0 = (int64_t)blockIdx.y * kTr;
#pragma unroll 4
    for (int i = ty; i < kTr; i += 4) {
        const int64_t t = t0 + i;
        tile[i][tx] = t < T ? X[t * ldx + k0 + tx] : (uint16_t)0;
    }
    __syncthreads();
#pragma unroll 4
    for (int i = ty; i < kTr; i += 4) {
        const int64_t t = t0 + tx;
        if (t < T_pad) Xt[(k0 + i) * T_pad + t] = tile[tx][i];
    }
}

}  // namespace

cudaError_t launch_transpose_x(const uint16_t* X, int64_t T, int64_t K, int64_t ldx,
                               uint16_t* Xt, int64_t T_pad, cudaStream_t st) {
    if (T <= 0 || K <= 0) return cudaSuccess;
    if (K % kTr || K / kTr > 65535) return cudaErrorInvalidValue;
    dim3 grid((unsigned)((T_pad + kTr - 1) / kTr), (unsigned)(K / kTr));
    transpose_x_kernel<<<grid, 256, 0, st>>>(X, T, K, ldx, Xt, T_pad);
    return cudaGetLastError();
}

}  // namespace awq
