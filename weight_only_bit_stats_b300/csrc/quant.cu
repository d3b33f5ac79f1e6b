// Candidate scales, INT4 packing and the search's final reduction.
//
// Method: "AWQ: Activation-aware Weight Quantization ..." (fdeinterviews.com
// /papers/awq), third paragraph: s is each channel's average activation
// magnitude raised to a power alpha, alpha from a grid search; every weight
// stays in low bits.  Last paragraph: 4 bits.  Asymmetric levels 0..15 per
// group of 128 with fp16 scale/zero are the library's stated format.
#include "common.cuh"
#include "kernels.cuh"
#include "int3.cuh"

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

// Eight lanes per (row, group), four row-groups per warp: lane c holds the
// 16 channels 16c..16c+15 of its row-group, forms the group's range with
// three shuffle rounds, rounds its 16 levels with the branch-free exact
// quotient (the same levels as the search producer's), and writes its two
// packed words; the eight lanes of a row-group write its 64 bytes at once.
__global__ void __launch_bounds__(256)
    pack_int4_kernel(const uint16_t* __restrict__ W, int64_t N, int64_t K, int64_t ldw,
                     const float* __restrict__ s, uint32_t* __restrict__ qweight,
                     uint16_t* __restrict__ scales, uint16_t* __restrict__ zeros,
                     unsigned* status) {
    const int lane = threadIdx.x & 31, c = lane & 7, rg = lane >> 3;
    const int64_t G = K / kGroup;
    const int64_t total = N * G;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    bool bad = false;
    // every lane runs the same number of iterations (the shuffles and the
    // vote need the whole warp); lanes past the end work on a clamped item
    for (int64_t base = warp0 * 4; base < total; base += nwarps * 4) {
        const int64_t item = base + rg;
        const bool live = item < total;
        const int64_t it = live ? item : total - 1;
        const int64_t n = it / G, g = it - n * G;
        const int64_t k0 = g * kGroup + 16 * c;
        const uint4* wp4 = reinterpret_cast<const uint4*>(W + n * ldw + k0);
        const uint4 r0 = __ldg(wp4), r1 = __ldg(wp4 + 1);
        float4 sv[4];
        if (s) {
            const float4* sp = reinterpret_cast<const float4*>(s + k0);
#pragma unroll
            for (int j = 0; j < 4; ++j) sv[j] = __ldg(sp + j);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) sv[j] = make_float4(1.f, 1.f, 1.f, 1.f);
        }
        const uint32_t wr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const float* sf = reinterpret_cast<const float*>(sv);
        float wp[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const uint32_t h = (wr[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
            wp[e] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)h)), sf[e]);
        }
        float lo = wp[0], hi = wp[0];
#pragma unroll
        for (int e = 1; e < 16; ++e) {
            lo = fmin_nan(lo, wp[e]);
            hi = fmax_nan(hi, wp[e]);
        }
        // this lane's 16 values: NaN or Inf makes lo or hi non-finite
        const bool lane_bad = !(isfinite(lo) && isfinite(hi));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        const GroupQuant gq = group_quant_from_range(lo, hi);
        if (live) bad |= lane_bad || !gq.finite;
        float rt[16];
        rint_quot8(wp, gq.scale, gq.rcp, rt);
        rint_quot8(wp + 8, gq.scale, gq.rcp, rt + 8);
        uint32_t w0 = 0, w1 = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            w0 |= (uint32_t)fminf(fmaxf(__fadd_rn(rt[e], gq.zf), 0.0f), 15.0f) << (4 * e);
            w1 |= (uint32_t)fminf(fmaxf(__fadd_rn(rt[e + 8], gq.zf), 0.0f), 15.0f) << (4 * e);
        }
        if (live) {
            *reinterpret_cast<uint2*>(qweight + n * (K / 8) + g * 16 + 2 * c) = make_uint2(w0, w1);
            if (c == 0) {
                scales[n * G + g] = __half_as_ushort(gq.scale_h);
                zeros[n * G + g] = __half_as_ushort(__float2half_rn(gq.zf));
            }
        }
    }
    if (bad) set_status(status, kStatusNonFinite);
}

// Group parameters at 3 bits: the rule of group_quant_from_range with the
// top level 7 instead of 15 (d = fp32(range / 7), zero-point clamped to 0..7).
// The exact-quotient rounding holds unchanged: only quotients below 8 in
// magnitude can leave the clamp.
__device__ __forceinline__ GroupQuant group_quant3_from_range(float lo, float hi) {
    GroupQuant g;
    const float range = __fsub_rn(hi, lo);
    float d = __fdiv_rn(range, 7.0f);
    d = fmaxf(d, 6.103515625e-05f);              // 2^-14, least normal fp16
    g.scale_h = __float2half_rn(d);
    g.scale = __half2float(g.scale_h);
    g.finite = isfinite(g.scale);
    g.rcp = __frcp_rn(g.scale);
    const float z = rint_quot(-lo, g.scale, g.rcp);
    g.zf = z > 0.0f ? fminf(z, 7.0f) : 0.0f;
    return g;
}

// 3-bit pack ("3 and 4 bits", AWQ page, fourth paragraph): the layout of
// pack_int4_kernel's lanes (8 per row-group, 16 channels each), levels
// 0..7, and three bit planes per 32 levels.  A lane sets bit p of its 16
// levels in the low or high half of plane word p; the lane pair of a 32-level
// block ORs its halves and the even lane writes the block's three words.
__global__ void __launch_bounds__(256)
    pack_int3_kernel(const uint16_t* __restrict__ W, int64_t N, int64_t K, int64_t ldw,
                     const float* __restrict__ s, uint32_t* __restrict__ planes,
                     uint16_t* __restrict__ scales, uint16_t* __restrict__ zeros,
                     unsigned* status) {
    const int lane = threadIdx.x & 31, c = lane & 7, rg = lane >> 3;
    const int64_t G = K / kGroup;
    const int64_t total = N * G;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    bool bad = false;
    for (int64_t base = warp0 * 4; base < total; base += nwarps * 4) {
        const int64_t item = base + rg;
        const bool live = item < total;
        const int64_t it = live ? item : total - 1;
        const int64_t n = it / G, g = it - n * G;
        const int64_t k0 = g * kGroup + 16 * c;
        const uint4* wp4 = reinterpret_cast<const uint4*>(W + n * ldw + k0);
        const uint4 r0 = __ldg(wp4), r1 = __ldg(wp4 + 1);
        float4 sv[4];
        if (s) {
            const float4* sp = reinterpret_cast<const float4*>(s + k0);
#pragma unroll
            for (int j = 0; j < 4; ++j) sv[j] = __ldg(sp + j);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) sv[j] = make_float4(1.f, 1.f, 1.f, 1.f);
        }
        const uint32_t wr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        const float* sf = reinterpret_cast<const float*>(sv);
        float wp[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const uint32_t h = (wr[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
            wp[e] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)h)), sf[e]);
        }
        float lo = wp[0], hi = wp[0];
#pragma unroll
        for (int e = 1; e < 16; ++e) {
            lo = fmin_nan(lo, wp[e]);
            hi = fmax_nan(hi, wp[e]);
        }
        const bool lane_bad = !(isfinite(lo) && isfinite(hi));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        const GroupQuant gq = group_quant3_from_range(lo, hi);
        if (live) bad |= lane_bad || !gq.finite;
        float rt[16];
        rint_quot8(wp, gq.scale, gq.rcp, rt);
        rint_quot8(wp + 8, gq.scale, gq.rcp, rt + 8);
        uint32_t p0 = 0, p1 = 0, p2 = 0;
        const int sh = 16 * (c & 1);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const uint32_t q = (uint32_t)fminf(fmaxf(__fadd_rn(rt[e], gq.zf), 0.0f), 7.0f);
            p0 |= (q & 1u) << (sh + e);
            p1 |= ((q >> 1) & 1u) << (sh + e);
            p2 |= (q >> 2) << (sh + e);
        }
        p0 |= __shfl_xor_sync(0xffffffffu, p0, 1);
        p1 |= __shfl_xor_sync(0xffffffffu, p1, 1);
        p2 |= __shfl_xor_sync(0xffffffffu, p2, 1);
        if (live) {
            if ((c & 1) == 0) {
                uint32_t* w = planes + n * (K / 32 * 3) + g * 12 + (c >> 1) * 3;
                w[0] = p0;
                w[1] = p1;
                w[2] = p2;
            }
            if (c == 0) {
                scales[n * G + g] = __half_as_ushort(gq.scale_h);
                zeros[n * G + g] = __half_as_ushort(__float2half_rn(gq.zf));
            }
        }
    }
    if (bad) set_status(status, kStatusNonFinite);
}

// mse[a] = (sum of alpha a's partials) / (T N): one warp per alpha, lane-
// strided fp64 sums added in a fixed butterfly order (deterministic); then
// the first argmin and its candidate scales.
__global__ void __launch_bounds__(256)
    search_finalize_kernel(const double* __restrict__ partials, int n_alpha, int64_t n_part,
                           int64_t T, int64_t N, int64_t K, const float* __restrict__ s_alpha,
                           double* __restrict__ mse, int32_t* __restrict__ best_idx,
                           float* __restrict__ s_out) {
    __shared__ double smse[64];
    __shared__ int sbest;
    const double denom = (double)T * (double)N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int a = warp; a < n_alpha; a += blockDim.x >> 5) {
        const double* pa = partials + (int64_t)a * n_part;
        double acc = 0.0;
        for (int64_t i = lane; i < n_part; i += 32) acc += pa[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            smse[a] = acc / denom;
            if (mse) mse[a] = acc / denom;
        }
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
    const float4* src = reinterpret_cast<const float4*>(s_alpha + (int64_t)sbest * K);
    float4* dst = reinterpret_cast<float4*>(s_out);
    for (int64_t k = threadIdx.x; k < K / 4; k += blockDim.x) dst[k] = src[k];
}

// Xs = fp16(fp32(X) * inv_s), 8 activations per thread (K % 8 == 0).
__global__ void __launch_bounds__(256)
    scale_x_kernel(const uint16_t* __restrict__ X, int64_t M, int64_t K, int64_t ldx,
                   const float* __restrict__ inv_s, uint16_t* __restrict__ Xs) {
    const int64_t per_row = K / 8, total = M * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = i / per_row, k = (i - m * per_row) * 8;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(X + m * ldx + k));
        const float4 a = __ldg(reinterpret_cast<const float4*>(inv_s + k));
        const float4 b = __ldg(reinterpret_cast<const float4*>(inv_s + k) + 1);
        const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
            const __half2 r = __floats2half2_rn(__fmul_rn(__low2float(h), f[2 * j]),
                                                __fmul_rn(__high2float(h), f[2 * j + 1]));
            w[j] = *reinterpret_cast<const uint32_t*>(&r);
        }
        *reinterpret_cast<uint4*>(Xs + m * K + k) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

cudaError_t launch_scale_x(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                           const float* inv_s, uint16_t* Xs, int num_sms, cudaStream_t st) {
    const int64_t total = M * (K / 8);
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    scale_x_kernel<<<(unsigned)blocks, 256, 0, st>>>(X, M, K, ldx, inv_s, Xs);
    return cudaGetLastError();
}

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
    int64_t blocks = (items + 31) / 32;               // 8 warps x 4 row-groups
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    pack_int4_kernel<<<(unsigned)blocks, 256, 0, st>>>(W, N, K, ldw, s, qweight, scales, zeros,
                                                       status);
    return cudaGetLastError();
}

cudaError_t launch_pack_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                             uint32_t* planes, uint16_t* scales, uint16_t* zeros, unsigned* status,
                             int num_sms, cudaStream_t st) {
    const int64_t items = N * (K / kGroup);
    if (items == 0) return cudaSuccess;
    int64_t blocks = (items + 31) / 32;               // 8 warps x 4 row-groups
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    pack_int3_kernel<<<(unsigned)blocks, 256, 0, st>>>(W, N, K, ldw, s, planes, scales, zeros,
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
