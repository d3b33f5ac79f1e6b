// W3A16 decode matmul for M <= 16 tokens over the 3-bit bit-plane format:
// Y[M,N] = X[M,K] deq(Wq)^T, deq = (q - z) * scale, fp32 accumulation.
//
// The pages evaluate the method at 3 bits as well as 4 ("AWQ: Activation-
// aware Weight Quantization ...", fdeinterviews.com/papers/awq, fourth
// paragraph) and note that fewer bytes per weight mean faster decoding
// (sixth paragraph).  Two kernels:
//
// gemv_w3a16_mma_kernel (when the activations fit in shared memory):
//  * One CTA per 16-row slab; its 8 warps split K by whole groups, and their
//    partial sums are added in warp order through shared memory.
//  * Levels i and i + 16 of a 32-level block sit at bits i and i + 16 of
//    each plane word: a rotate and a LOP3 per plane place both under the
//    mantissa of fp16 1024, and one HSUB2 gives the exact pair (q - z).
//    Lane t of a row builds the pairs i = t, t + 4, t + 8, t + 12, which are
//    exactly its A fragments of two mma.m16n8k16 (the MMA's k order is a
//    permutation of the block's levels), so the products go to the tensor
//    cores in fp32.  The activations are staged once per CTA in the same
//    permuted order; each group's sums get the group scale in fp32.
//
// gemv_w3a16_kernel (any size):
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

// ---- tensor-core kernel ----
constexpr int kW3mWarps = 8;
constexpr size_t kW3mSmemMax = 200 * 1024;

__device__ __forceinline__ uint32_t rotr(uint32_t w, uint32_t n) { return __funnelshift_r(w, w, n); }

__device__ __forceinline__ uint32_t lop3_or(uint32_t a, uint32_t mask, uint32_t c) {
    uint32_t d;      // (a & mask) | c
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
    return d;
}

// Exact fp16 pair (q_i - z, q_{i+16} - z) of one block, rotations r0..r2 =
// (i - p) mod 32 for plane p.
__device__ __forceinline__ uint32_t pair_mz(uint32_t p0, uint32_t p1, uint32_t p2, uint32_t r0,
                                            uint32_t r1, uint32_t r2, __half2 z1024) {
    uint32_t v = lop3_or(rotr(p0, r0), 0x00010001u, 0x64006400u);
    v = lop3_or(rotr(p1, r1), 0x00020002u, v);
    v = lop3_or(rotr(p2, r2), 0x00040004u, v);
    const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&v), z1024);
    return *reinterpret_cast<const uint32_t*>(&d);
}

__device__ __forceinline__ void mma16816_3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared activations: per token a row of K*2 + 64 bytes (the pad puts
// consecutive tokens on different bank halves); block j's 64 bytes hold,
// for t = 0..3, x[32j+t+{0,16,4,20,8,24,12,28}] -- lane t's two B fragments
// of each of the block's two MMAs.
__host__ __device__ constexpr int64_t w3_x_row_bytes(int64_t K) { return K * 2 + 64; }

template <int NB>
__global__ void __launch_bounds__(kW3mWarps * 32)
    gemv_w3a16_mma_kernel(const uint16_t* __restrict__ X, int64_t ldx, int M,
                          const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                          const uint16_t* __restrict__ zeros, int64_t N, int64_t K,
                          uint16_t* __restrict__ Y, int64_t ldy) {
    constexpr int kCols = 8 * NB;
    extern __shared__ __align__(16) uint8_t w3_smem[];
    const int64_t xrow = w3_x_row_bytes(K);
    float* part = reinterpret_cast<float*>(w3_smem + (int64_t)M * xrow);  // [warp][16][kCols]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int64_t nbk = K / 32, G = K / kGroup;

    // stage the activations in fragment order
    for (int64_t idx = threadIdx.x; idx < (int64_t)M * nbk * 4; idx += kW3mWarps * 32) {
        const int64_t m = idx / (nbk * 4), rem = idx - m * nbk * 4;
        const int64_t j = rem >> 2;
        const int tt = (int)(rem & 3);
        const uint16_t* xs = X + m * ldx + 32 * j + tt;
        const uint32_t w0 = (uint32_t)__ldg(xs) | ((uint32_t)__ldg(xs + 16) << 16);
        const uint32_t w1 = (uint32_t)__ldg(xs + 4) | ((uint32_t)__ldg(xs + 20) << 16);
        const uint32_t w2 = (uint32_t)__ldg(xs + 8) | ((uint32_t)__ldg(xs + 24) << 16);
        const uint32_t w3 = (uint32_t)__ldg(xs + 12) | ((uint32_t)__ldg(xs + 28) << 16);
        *reinterpret_cast<uint4*>(w3_smem + m * xrow + j * 64 + tt * 16) = make_uint4(w0, w1, w2, w3);
    }
    __syncthreads();

    const int64_t row_a = (int64_t)blockIdx.x * 16 + g, row_b = row_a + 8;
    const bool va = row_a < N, vb = row_b < N;
    const uint4* pa = reinterpret_cast<const uint4*>(planes + (va ? row_a : 0) * nbk * 3);
    const uint4* pb = reinterpret_cast<const uint4*>(planes + (vb ? row_b : 0) * nbk * 3);
    const uint8_t* xs[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) xs[nb] = w3_smem + min(g + 8 * nb, M - 1) * xrow + t * 16;
    // rotations for the pairs i = t + 4c, plane p: (t + 4c - p) mod 32
    uint32_t rot[4][3];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int p = 0; p < 3; ++p) rot[c][p] = (uint32_t)(t + 4 * c - p) & 31u;

    float y[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int k = 0; k < 4; ++k) y[nb][k] = 0.0f;
    const int g0 = (int)((int64_t)warp * G / kW3mWarps), g1 = (int)((int64_t)(warp + 1) * G / kW3mWarps);
    for (int gi = g0; gi < g1; ++gi) {
        uint4 wa[3], wb[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            wa[k] = va ? __ldg(pa + gi * 3 + k) : make_uint4(0, 0, 0, 0);
            wb[k] = vb ? __ldg(pb + gi * 3 + k) : make_uint4(0, 0, 0, 0);
        }
        const float sa = va ? __half2float(__ushort_as_half(__ldg(scales + row_a * G + gi))) : 0.0f;
        const float sb = vb ? __half2float(__ushort_as_half(__ldg(scales + row_b * G + gi))) : 0.0f;
        const __half h1024 = __float2half_rn(1024.0f);
        const __half2 za = __half2half2(
            __hadd(h1024, __ushort_as_half(va ? __ldg(zeros + row_a * G + gi) : (uint16_t)0)));
        const __half2 zb = __half2half2(
            __hadd(h1024, __ushort_as_half(vb ? __ldg(zeros + row_b * G + gi) : (uint16_t)0)));
        const uint32_t A[12] = {wa[0].x, wa[0].y, wa[0].z, wa[0].w, wa[1].x, wa[1].y,
                                wa[1].z, wa[1].w, wa[2].x, wa[2].y, wa[2].z, wa[2].w};
        const uint32_t B[12] = {wb[0].x, wb[0].y, wb[0].z, wb[0].w, wb[1].x, wb[1].y,
                                wb[1].z, wb[1].w, wb[2].x, wb[2].y, wb[2].z, wb[2].w};
        float cacc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int k = 0; k < 4; ++k) cacc[nb][k] = 0.0f;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            const uint32_t a0 = A[3 * blk], a1 = A[3 * blk + 1], a2 = A[3 * blk + 2];
            const uint32_t b0 = B[3 * blk], b1 = B[3 * blk + 1], b2 = B[3 * blk + 2];
            uint32_t fa[4], fb[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                fa[c] = pair_mz(a0, a1, a2, rot[c][0], rot[c][1], rot[c][2], za);
                fb[c] = pair_mz(b0, b1, b2, rot[c][0], rot[c][1], rot[c][2], zb);
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const uint4 xb = *reinterpret_cast<const uint4*>(xs[nb] + ((int64_t)gi * 4 + blk) * 64);
                mma16816_3(cacc[nb], fa[0], fb[0], fa[1], fb[1], xb.x, xb.y);
                mma16816_3(cacc[nb], fa[2], fb[2], fa[3], fb[3], xb.z, xb.w);
            }
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            y[nb][0] = fmaf(sa, cacc[nb][0], y[nb][0]);
            y[nb][1] = fmaf(sa, cacc[nb][1], y[nb][1]);
            y[nb][2] = fmaf(sb, cacc[nb][2], y[nb][2]);
            y[nb][3] = fmaf(sb, cacc[nb][3], y[nb][3]);
        }
    }
    // this warp's partial sums, then the warps' sums in warp order
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int row = g + (k < 2 ? 0 : 8), col = nb * 8 + 2 * t + (k & 1);
            part[(warp * 16 + row) * kCols + col] = y[nb][k];
        }
    __syncthreads();
    for (int e = threadIdx.x; e < 16 * M; e += kW3mWarps * 32) {
        const int row = e & 15, m = e >> 4;
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < kW3mWarps; ++w) acc += part[(w * 16 + row) * kCols + m];
        const int64_t n = (int64_t)blockIdx.x * 16 + row;
        if (n < N) Y[(int64_t)m * ldy + n] = __half_as_ushort(__float2half_rn(acc));
    }
}

template <int NB>
cudaError_t launch_mma(const uint16_t* X, int64_t ldx, int M, const uint32_t* planes,
                       const uint16_t* scales, const uint16_t* zeros, int64_t N, int64_t K,
                       uint16_t* Y, int64_t ldy, size_t smem, cudaStream_t st) {
    cudaError_t e = smem_attr_once<gemv_w3a16_mma_kernel<NB>>((int)kW3mSmemMax);
    if (e != cudaSuccess) return e;
    const int64_t slabs = (N + 15) / 16;
    gemv_w3a16_mma_kernel<NB><<<(unsigned)slabs, kW3mWarps * 32, smem, st>>>(
        X, ldx, M, planes, scales, zeros, N, K, Y, ldy);
    return cudaGetLastError();
}

// ---- CUDA-core kernel ----
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
    // the tensor-core kernel when the activations fit in shared memory (and
    // the planes allow 16-byte loads)
    const size_t smem = (size_t)M * (size_t)w3_x_row_bytes(K) +
                        (size_t)kW3mWarps * 16 * (M <= 8 ? 8 : 16) * sizeof(float);
    if (smem <= kW3mSmemMax && (reinterpret_cast<uintptr_t>(planes) & 15u) == 0)
        return M <= 8 ? launch_mma<1>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, smem, st)
                      : launch_mma<2>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, smem, st);
    if (M == 1) return launch_mt<1>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, num_sms, st);
    if (M <= 4) return launch_mt<4>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, num_sms, st);
    if (M <= 8) return launch_mt<8>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, num_sms, st);
    return launch_mt<16>(X, ldx, M, planes, scales, zeros, N, K, Y, ldy, num_sms, st);
}

}  // namespace awq
