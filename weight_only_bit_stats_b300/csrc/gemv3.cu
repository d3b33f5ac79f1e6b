// W3A16 decode matmul for M <= 16 tokens over the 3-bit bit-plane format:
// Y[M,N] = X[M,K] deq(Wq)^T, deq = (q - z) * scale, fp32 accumulation.
//
// The pages evaluate the method at 3 bits as well as 4 ("AWQ: Activation-
// aware Weight Quantization ...", fdeinterviews.com/papers/awq, fourth
// paragraph) and note that fewer bytes per weight mean faster decoding
// (sixth paragraph).  This first 3-bit kernel is plain CUDA-core code:
//
//  * One warp per output row at a time; lane l takes the row's 32-level
//    blocks l, l + 32, ..., four at a time: the plane words, scales and
//    zero-points of four blocks are requested before any is used, so a row
//    costs one memory round trip per four blocks rather than per block.
//  * Levels i and i + 16 of a block sit at bits i and i + 16 of each plane,
//    so three shifts and three LOP3s place both levels' bits under the
//    mantissa of fp16 1024 at once; one HSUB2 gives the exact pair
//    (q - z), which is widened and scaled to the exact fp32 values
//    (q - z) * scale (at most 3 + 11 significant bits) and multiplied into
//    every token's accumulator with fp32 FMAs.  The activations come
//    through L1 as 16-byte loads.
//  * The 32 lanes' sums are added in a fixed butterfly order, so the result
//    is deterministic.
#include "common.cuh"
#include "int3.cuh"

namespace awq {
namespace {

constexpr int kW3Warps = 8;
constexpr int kW3Batch = 4;                  // blocks a lane loads at once

__device__ __forceinline__ uint32_t lop3_or_and(uint32_t a, uint32_t mask, uint32_t c) {
    uint32_t d;      // (a & mask) | c
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
    return d;
}

// Bits i and i + 16 of plane p, moved to bits p and 16 + p.
template <int I, int P>
__device__ __forceinline__ uint32_t plane_bits(uint32_t w) {
    if constexpr (I >= P) return w >> (I - P);
    else return w << (P - I);
}

// The exact fp32 weights (q - z) * sc of levels I and I + 16 of a block.
template <int I>
__device__ __forceinline__ void level_pair(uint32_t p0, uint32_t p1, uint32_t p2,
                                           __half2 z1024, float sc, float& wa, float& wb) {
    uint32_t v = lop3_or_and(plane_bits<I, 0>(p0), 0x00010001u, 0x64006400u);
    v = lop3_or_and(plane_bits<I, 1>(p1), 0x00020002u, v);
    v = lop3_or_and(plane_bits<I, 2>(p2), 0x00040004u, v);
    const float2 d = __half22float2(__hsub2(*reinterpret_cast<const __half2*>(&v), z1024));
    wa = __fmul_rn(d.x, sc);
    wb = __fmul_rn(d.y, sc);
}

template <int I>
__device__ __forceinline__ void block_weights(uint32_t p0, uint32_t p1, uint32_t p2,
                                              __half2 z1024, float sc, float (&w)[32]) {
    if constexpr (I < 16) {
        level_pair<I>(p0, p1, p2, z1024, sc, w[I], w[I + 16]);
        block_weights<I + 1>(p0, p1, p2, z1024, sc, w);
    }
}

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
        for (int64_t j0 = lane; j0 < nb; j0 += 32 * kW3Batch) {
            uint32_t pw[kW3Batch][3];
            uint16_t sb[kW3Batch], zb[kW3Batch];
#pragma unroll
            for (int b = 0; b < kW3Batch; ++b) {
                const int64_t j = j0 + 32 * b;
                if (j < nb) {
                    pw[b][0] = __ldg(prow + j * 3);
                    pw[b][1] = __ldg(prow + j * 3 + 1);
                    pw[b][2] = __ldg(prow + j * 3 + 2);
                    sb[b] = __ldg(scales + n * G + (j >> 2));   // 4 blocks per group
                    zb[b] = __ldg(zeros + n * G + (j >> 2));
                }
            }
#pragma unroll
            for (int b = 0; b < kW3Batch; ++b) {
            const int64_t j = j0 + 32 * b;
            if (j >= nb) break;
            const float sc = __half2float(__ushort_as_half(sb[b]));
            const __half2 z1024 =
                __half2half2(__hadd(__float2half_rn(1024.0f), __ushort_as_half(zb[b])));
            float w[32];
            block_weights<0>(pw[b][0], pw[b][1], pw[b][2], z1024, sc, w);
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
