// W3A16 decode matmul for M <= 16 tokens over the 3-bit bit-plane format:
// Y[M,N] = X[M,K] deq(Wq)^T, deq = (q - z) * scale, fp32 accumulation.
//
// The pages evaluate the method at 3 bits as well as 4 ("AWQ: Activation-
// aware Weight Quantization ...", fdeinterviews.com/papers/awq, fourth
// paragraph) and note that fewer bytes per weight mean faster decoding
// (sixth paragraph).  This first 3-bit kernel is plain CUDA-core code:
//
//  * One warp per output row at a time; lane l takes the row's 32-level
//    blocks l, l + 32, ... (three plane words each, three coalesced 4-byte
//    loads per warp step).
//  * A block's 32 levels are rebuilt from the three planes, turned into the
//    exact fp32 values (q - z) * scale (at most 3 + 11 significant bits),
//    and multiplied into every token's accumulator with fp32 FMAs; the
//    activations come through L1 as 16-byte loads.
//  * The 32 lanes' sums are added in a fixed butterfly order, so the result
//    is deterministic.
#include "common.cuh"
#include "int3.cuh"

namespace awq {
namespace {

constexpr int kW3Warps = 8;

template <int MT>
__global__ void __launch_bounds__(kW3Warps * 32, 2)
    gemv_w3a16_kernel(const uint16_t* __restrict__ X, int64_t ldx, int M,
                      const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                      const uint16_t* __restrict__ zeros, int64_t N, int64_t K,
                      uint16_t* __restrict__ Y, int64_t ldy) {
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / 32;                 // 32-level blocks per row
    const int64_t G = K / kGroup;
    const int64_t warp0 = (int64_t)blockIdx.x * kW3Warps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * kW3Warps;
    for (int64_t n = warp0; n < N; n += nwarps) {
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
        const uint32_t* prow = planes + n * nb * 3;
        for (int64_t j = lane; j < nb; j += 32) {
            const uint32_t p0 = __ldg(prow + j * 3);
            const uint32_t p1 = __ldg(prow + j * 3 + 1);
            const uint32_t p2 = __ldg(prow + j * 3 + 2);
            const int64_t g = j >> 2;              // 4 blocks per group of 128
            const float sc = __half2float(__ushort_as_half(__ldg(scales + n * G + g)));
            const float z = __half2float(__ushort_as_half(__ldg(zeros + n * G + g)));
            float w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const uint32_t q = ((p0 >> i) & 1u) | (((p1 >> i) & 1u) << 1) |
                                   (((p2 >> i) & 1u) << 2);
                w[i] = __fmul_rn(__fsub_rn((float)q, z), sc);   // exact
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < M) {
                    const uint4* xp = reinterpret_cast<const uint4*>(X + (int64_t)m * ldx + j * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint4 xv = __ldg(xp + v);
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const __half2 x2 = *reinterpret_cast<const __half2*>(&xw[h]);
                            acc[m] = fmaf(w[v * 8 + 2 * h], __low2float(x2), acc[m]);
                            acc[m] = fmaf(w[v * 8 + 2 * h + 1], __high2float(x2), acc[m]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float a = acc[m];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0 && m < M) Y[(int64_t)m * ldy + n] = __half_as_ushort(__float2half_rn(a));
        }
    }
}

template <int MT>
cudaError_t launch_mt(const uint16_t* X, int64_t ldx, int M, const uint32_t* planes,
                      const uint16_t* scales, const uint16_t* zeros, int64_t N, int64_t K,
                      uint16_t* Y, int64_t ldy, int num_sms, cudaStream_t st) {
    int64_t blocks = (N + kW3Warps - 1) / kW3Warps;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    gemv_w3a16_kernel<MT><<<(unsigned)blocks, kW3Warps * 32, 0, st>>>(X, ldx, M, planes, scales,
                                                                      zeros, N, K, Y, ldy);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_w3a16(const uint16_t* X, int64_t ldx, int M, const uint32_t* planes,
                              const uint16_t* scales, const uint16_t* zeros, int64_t N, int64_t K,
                              uint16_t* Y, int64_t ldy, int num_sms, cudaStream_t st) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (M == 1) return launch_mt<1>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, num_sms, st);
    if (M <= 4) return launch_mt<4>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, num_sms, st);
    if (M <= 8) return launch_mt<8>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, num_sms, st);
    return launch_mt<16>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, num_sms, st);
}

}  // namespace awq
