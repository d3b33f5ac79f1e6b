// Candidate scales, INT4 packing and the search's final reduction.
//
// Method: "AWQ: Activation-aware Weight Quantization ..." (fdeinterviews.com
// /papers/awq), third paragraph: s is each channel's average activation
// magnitude raised to a power alpha, alpha from a grid search; every weight
// stays in low bits.  Last paragraph: 4 bits.  Asymmetric levels 0..15 per
// group of 128 with fp16 scale/zero are the library's stated format.
#include "common.cuh"
#include "kernels.cuh"

namespace awq {
namespace {

constexpr int kCandThreads = 256;

// Pass 1: r_k = pow(max(m_k, 1e-4), alpha) and per-block max / min of r.
__global__ void __launch_bounds__(kCandThreads)
    cand_pass1_kernel(const double* __restrict__ mean, int64_t K, AlphaList alphas,
                      double* __restrict__ ws_r, double* __restrict__ ws_mm) {
    __shared__ double smax[kCandThreads / 32], smin[kCandThreads / 32];
    const int a = blockIdx.y;
    const int64_t k = (int64_t)blockIdx.x * kCandThreads + threadIdx.x;
    double r = 0.0, mx = -INFINITY, mn = INFINITY;
    if (k < K) {
        r = pow(fmax(mean[k], 1e-4), alphas.a[a]);
        ws_r[(int64_t)a * K + k] = r;
        mx = r;
        mn = r;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = fmin(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if ((threadIdx.x & 31) == 0) {
        smax[threadIdx.x >> 5] = mx;
        smin[threadIdx.x >> 5] = mn;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kCandThreads / 32; ++w) {
            mx = fmax(mx, smax[w]);
            mn = fmin(mn, smin[w]);
        }
        int64_t slot = ((int64_t)a * gridDim.x + blockIdx.x) * 2;
        ws_mm[slot] = mx;
        ws_mm[slot + 1] = mn;
    }
}

// Pass 2: s_k = fp32(r_k / sqrt(max r * min r)); also 1/s_k (IEEE fp32).
__global__ void __launch_bounds__(kCandThreads)
    cand_pass2_kernel(int64_t K, int n_blocks, const double* __restrict__ ws_r,
                      const double* __restrict__ ws_mm, float* __restrict__ s_alpha,
                      float* __restrict__ inv_s_alpha) {
    __shared__ double norm_s;
    const int a = blockIdx.y;
    if (threadIdx.x == 0) {
        double mx = -INFINITY, mn = INFINITY;
        for (int b = 0; b < n_blocks; ++b) {
            mx = fmax(mx, ws_mm[((int64_t)a * n_blocks + b) * 2]);
            mn = fmin(mn, ws_mm[((int64_t)a * n_blocks + b) * 2 + 1]);
        }
        norm_s = sqrt(mx * mn);
    }
    __syncthreads();
    const int64_t k = (int64_t)blockIdx.x * kCandThreads + threadIdx.x;
    if (k < K) {
        float s = __double2float_rn(ws_r[(int64_t)a * K + k] / norm_s);
        s_alpha[(int64_t)a * K + k] = s;
        if (inv_s_alpha) inv_s_alpha[(int64_t)a * K + k] = __frcp_rn(s);
    }
}

// One warp per (row, group): quantise 128 scaled weights and write 16 words,
// the group's fp16 scale and fp16 zero-point.
__global__ void __launch_bounds__(256)
    pack_int4_kernel(const uint16_t* __restrict__ W, int64_t N, int64_t K, int64_t ldw,
                     const float* __restrict__ s, uint32_t* __restrict__ qweight,
                     uint16_t* __restrict__ scales, uint16_t* __restrict__ zeros,
                     unsigned* status) {
    const int lane = threadIdx.x & 31;
    const int64_t G = K / kGroup;
    const int64_t total = N * G;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    bool bad = false;
    for (int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < total;
         item += nwarps) {
        const int64_t n = item / G, g = item - n * G;
        const int64_t k0 = g * kGroup + 4 * lane;
        uint2 raw = __ldg(reinterpret_cast<const uint2*>(W + n * ldw + k0));
        float4 sv = s ? __ldg(reinterpret_cast<const float4*>(s + k0)) : make_float4(1, 1, 1, 1);
        float wp[4];
        wp[0] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(raw.x & 0xFFFFu))), sv.x);
        wp[1] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(raw.x >> 16))), sv.y);
        wp[2] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(raw.y & 0xFFFFu))), sv.z);
        wp[3] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(raw.y >> 16))), sv.w);
        float lo = wp[0], hi = wp[0];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            bad |= !isfinite(wp[e]);
            lo = fminf(lo, wp[e]);
            hi = fmaxf(hi, wp[e]);
        }
        GroupQuant gq = group_quant_params(lo, hi);
        bad |= !gq.finite;
        uint32_t v = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) v |= (uint32_t)quant_level(wp[e], gq) << (4 * e);
        uint32_t other = __shfl_xor_sync(0xffffffffu, v, 1);
        if ((lane & 1) == 0) qweight[n * (K / 8) + g * 16 + (lane >> 1)] = v | (other << 16);
        if (lane == 0) {
            scales[n * G + g] = __half_as_ushort(gq.scale_h);
            zeros[n * G + g] = __half_as_ushort(__float2half_rn(gq.zf));
        }
    }
    if (bad) set_status(status, kStatusNonFinite);
}

__global__ void __launch_bounds__(256)
    search_finalize_kernel(const double* __restrict__ partials, int n_alpha, int64_t n_part,
                           int64_t T, int64_t N, int64_t K, const float* __restrict__ s_alpha,
                           double* __restrict__ mse, int32_t* __restrict__ best_idx,
                           float* __restrict__ s_out) {
    __shared__ double smse[64];
    __shared__ int sbest;
    const double denom = (double)T * (double)N;
    for (int a = threadIdx.x; a < n_alpha; a += blockDim.x) {
        double acc = 0.0;
        for (int64_t i = 0; i < n_part; ++i) acc += partials[(int64_t)a * n_part + i];
        smse[a] = acc / denom;
        if (mse) mse[a] = acc / denom;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int b = 0;
        for (int a = 1; a < n_alpha; ++a)
            if (smse[a] < smse[b]) b = a;
        sbest = b;
        *best_idx = b;
    }
    __syncthreads();
    const float* src = s_alpha + (int64_t)sbest * K;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) s_out[k] = src[k];
}

}  // namespace

int cand_blocks(int64_t K) { return (int)((K + kCandThreads - 1) / kCandThreads); }

cudaError_t launch_candidate_scales(const double* mean, int64_t K, const AlphaList& alphas,
                                    int n_alpha, float* s_alpha, float* inv_s_alpha, double* ws_r,
                                    double* ws_mm, cudaStream_t st) {
    dim3 grid(cand_blocks(K), n_alpha);
    cand_pass1_kernel<<<grid, kCandThreads, 0, st>>>(mean, K, alphas, ws_r, ws_mm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cand_pass2_kernel<<<grid, kCandThreads, 0, st>>>(K, cand_blocks(K), ws_r, ws_mm, s_alpha,
                                                      inv_s_alpha);
    return cudaGetLastError();
}

cudaError_t launch_pack_int4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                             uint32_t* qweight, uint16_t* scales, uint16_t* zeros, unsigned* status,
                             int num_sms, cudaStream_t st) {
    const int64_t items = N * (K / kGroup);
    if (items == 0) return cudaSuccess;
    int64_t blocks = (items + 7) / 8;
    const int64_t cap = (int64_t)num_sms * 16;
    if (blocks > cap) blocks = cap;
    pack_int4_kernel<<<(unsigned)blocks, 256, 0, st>>>(W, N, K, ldw, s, qweight, scales, zeros,
                                                       status);
    return cudaGetLastError();
}

cudaError_t launch_search_finalize(const double* partials, int n_alpha, int64_t n_part, int64_t T,
                                   int64_t N, int64_t K, const float* s_alpha, double* mse,
                                   int32_t* best_idx, float* s_out, cudaStream_t st) {
    search_finalize_kernel<<<1, 256, 0, st>>>(partials, n_alpha, n_part, T, N, K, s_alpha, mse,
                                              best_idx, s_out);
    return cudaGetLastError();
}

}  // namespace awq
