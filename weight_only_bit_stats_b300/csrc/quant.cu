// Candidate scales, INT4 packing and the search's final reduction.
//
// Method: "AWQ: Activation-aware Weight Quantization ..." (fdeinterviews.com
// /papers/awq), third paragraph: s is a power alpha of the channel's mean
// absolute activation, alpha is picked from a grid, and all stored weights
// are low-bit.  Last paragraph: 4 bits.  Asymmetric levels 0..15 per
// group of 128 with fp16 scale/zero are the library's stated format.
#include "common.cuh"
#include "kernels.cuh"
#include "int3.cuh"

namespace awq {
namespace {

// Candidate scales: pass 1 in blocks of 64 (the fp64 pow is the work; small
// blocks spread it evenly over the SMs), pass 2 in blocks of 256.
constexpr int kCandThreads = 64;
constexpr int kCand2Threads = 256;
// Pack launch shape: 128-thread blocks held to 96 registers (five resident
// per SM), grid capped at two waves of them.
#ifndef AWQ_PACK_BLOCKS_PER_SM
#define AWQ_PACK_BLOCKS_PER_SM 10
#endif
#ifndef AWQ_PACK_THREADS
#define AWQ_PACK_THREADS 128
#endif
#ifndef AWQ_PACK_MIN_BLOCKS
#define AWQ_PACK_MIN_BLOCKS 5
#endif
constexpr int kPackBlocksPerSm = AWQ_PACK_BLOCKS_PER_SM;
constexpr int kPackThreads = AWQ_PACK_THREADS;
constexpr int kPackMinBlocks = AWQ_PACK_MIN_BLOCKS;

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
// The first warp reduces pass 1's block extremes (max and min are exact,
// so the order does not matter).
__global__ void __launch_bounds__(kCand2Threads)
    cand_pass2_kernel(int64_t K, int n_blocks, const double* __restrict__ ws_r,
                      const double* __restrict__ ws_mm, float* __restrict__ s_alpha,
                      float* __restrict__ inv_s_alpha) {
    __shared__ double norm_s;
    const int a = blockIdx.y;
    if (threadIdx.x < 32) {
        double mx = -INFINITY, mn = INFINITY;
        for (int b = threadIdx.x; b < n_blocks; b += 32) {
            mx = fmax(mx, ws_mm[((int64_t)a * n_blocks + b) * 2]);
            mn = fmin(mn, ws_mm[((int64_t)a * n_blocks + b) * 2 + 1]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fmin(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        if (threadIdx.x == 0) norm_s = sqrt(mx * mn);
    }
    __syncthreads();
    const int64_t k = (int64_t)blockIdx.x * kCand2Threads + threadIdx.x;
    if (k < K) {
        float s = __double2float_rn(ws_r[(int64_t)a * K + k] / norm_s);
        s_alpha[(int64_t)a * K + k] = s;
        if (inv_s_alpha) inv_s_alpha[(int64_t)a * K + k] = __frcp_rn(s);
    }
}

// Level bits without a float-to-integer conversion: for an integer-valued
// rt (or +-Inf, NaN, or any magnitude), fp32 min(max(rt + (z + 2^23), 2^23),
// qmax + 2^23) is 2^23 + clamp(rt + z, 0, qmax) exactly (the sums are exact
// below 2^24 in magnitude and rounding is monotone above), and its bit
// pattern is 0x4B000000 + level.  Summing (0x4B000000 + L_e) 16^e over eight
// levels modulo 2^32 leaves sum L_e 16^e plus 0x4B000000 + 0xB0000000 (the
// higher terms of the constant vanish).
__device__ __forceinline__ uint32_t nibbles8_exact(const float* wp, float scale, float rcp,
                                                   float zf, float qmax) {
    const float zb = __fadd_rn(zf, 8388608.0f), topb = qmax + 8388608.0f;
    uint32_t acc = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float t0 = __fmul_rn(wp[e], rcp);
        float rt = rint_small(t0);
        if (near_tie(t0, rt)) rt = rintf(__fdiv_rn(wp[e], scale));
        acc += __float_as_uint(fminf(fmaxf(__fadd_rn(rt, zb), 8388608.0f), topb)) << (4 * e);
    }
    return acc - 0xFB000000u;
}

// Bit p of each of the 8 nibbles of w, as 8 contiguous bits.
__device__ __forceinline__ uint32_t nibble_plane(uint32_t w, int p) {
    uint32_t x = (w >> p) & 0x11111111u;
    x = (x | (x >> 3)) & 0x03030303u;
    x = (x | (x >> 6)) & 0x000F000Fu;
    return (x | (x >> 12)) & 0xFFu;
}

// The fast levels of 32 scaled weights (16 pairs) as four nibble words
// (eight levels each), and whether any quotient came near a tie.  y =
// fp32(t + 1.5 * 2^23) holds rint(t) in its low mantissa bits for |t| <
// 2^22: with t clamped to [-z, qmax - z] (CLAMP), or known to round inside
// it, the bit pattern of y is 0x4B400000 + rint(t), so the level rint(t) + z
// is the pattern minus 0x4B400000 - z.  Clamping t before rounding equals
// clamping after, the bounds being integers; a clamped t is an integer and
// is never near a tie.  The pair operations round each lane as the scalar
// ones do.
template <bool CLAMP>
__device__ __forceinline__ bool fast_nibbles32(const float2* wp, float rcp, float zf, float qmax,
                                               uint32_t* w) {
    const float kM = 12582912.0f;               // 1.5 * 2^23
    const float2 rcp2 = make_float2(rcp, rcp), m2 = make_float2(kM, kM);
    const float2 negm2 = make_float2(-kM, -kM), neg1 = make_float2(-1.0f, -1.0f);
    const float lo = -zf, hi = qmax - zf;
    const uint32_t bias = (0x4B400000u - (uint32_t)zf) * 0x11111111u;
    float dmax[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t acc = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float2 t = __fmul2_rn(wp[4 * i + e], rcp2);
            if (CLAMP) {
                t.x = fminf(fmaxf(t.x, lo), hi);
                t.y = fminf(fmaxf(t.y, lo), hi);
            }
            const float2 y = __fadd2_rn(t, m2);
            const float2 d = __ffma2_rn(__fadd2_rn(y, negm2), neg1, t);   // t - rint(t)
            dmax[e] = fmaxf(dmax[e], fmaxf(fabsf(d.x), fabsf(d.y)));
            acc += __float_as_uint(y.x) << (8 * e);
            acc += __float_as_uint(y.y) << (8 * e + 4);
        }
        w[i] = acc - bias;
    }
    return fmaxf(fmaxf(dmax[0], dmax[1]), fmaxf(dmax[2], dmax[3])) > kTieBand;
}

// Four lanes per (row, group), eight row-groups per warp.  A row-group is
// 16 chunks of 8 channels (16 bytes of W each); lane c holds chunks 4j + c,
// j = 0..3, so each of its four 16-byte loads reads 64 contiguous bytes of
// the row across the four lanes.  A warp's unit is eight consecutive rows of
// one group g: the warp stages s for g in its own shared-memory slice (one
// 512-byte load), which the eight row-groups then read as broadcasts.  Units
// are walked with a fixed stride kept as a quotient and remainder of G, so
// that no iteration divides.
//
// The group's range takes two shuffle rounds; the 32 levels of a lane use
// the branch-free exact quotient (the same levels as the search producer's).
// When rint(lo / d) and rint(hi / d) (the fast quotients of the group's
// extremes; every quotient of the group lies between them) already fall in
// [-z, qmax - z] for every row-group of the warp, no level can leave 0..qmax
// and the clamp is skipped.  When any quotient of the warp comes near a tie,
// the warp recomputes its levels with the exact quotient.
//
// BITS = 4: chunk 4j + c is packed word 4j + c of the row-group.  BITS = 3
// (the AWQ page, fourth paragraph, evaluates 3 and 4 bits): levels 0..7 in
// three bit planes per 32-level block; block j is chunks 4j..4j+3, one per
// lane, so the lanes' plane bytes are transposed across the four lanes (two
// shuffle rounds with byte permutes) and lane c writes block c's three words.
template <int BITS>
__global__ void __launch_bounds__(kPackThreads, kPackMinBlocks)
    pack_kernel(const uint16_t* __restrict__ W, int64_t N, int64_t K, int64_t ldw,
                const float* __restrict__ s, uint32_t* __restrict__ out,
                uint16_t* __restrict__ scales, uint16_t* __restrict__ zeros, unsigned* status) {
    constexpr float kQmax = (float)((1 << BITS) - 1);
    __shared__ __align__(16) float s_sh[kPackThreads / 32][kGroup];
    const int lane = threadIdx.x & 31, c = lane & 3, rg = lane >> 2;
    float* ss = s_sh[threadIdx.x >> 5];
    const int64_t G = K / kGroup;
    const int64_t chunks = (N + 7) / 8, units = chunks * G;
    const int64_t unit0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t sq = stride / G, sr = stride - sq * G;
    int64_t chunk = unit0 / G, g = unit0 - chunk * G;
    // byte-transpose selectors of the 3-bit planes (lane-dependent)
    const uint32_t sel2 = (c & 2) ? 0x3276u : 0x5410u, sel1 = (c & 1) ? 0x3715u : 0x6240u;
    // unit (chunk, g) -> this lane's four 16-byte pieces of W and the warp's
    // 512-byte piece of s for g (rows past N - 1 read row N - 1)
    auto fetch = [&](int64_t ch, int64_t gg, uint4* raw, float4& sv) {
        const int64_t n = ch * 8 + rg;
        const uint4* wp4 = reinterpret_cast<const uint4*>(W + (n < N ? n : N - 1) * ldw + gg * kGroup);
#pragma unroll
        for (int j = 0; j < 4; ++j) raw[j] = __ldg(wp4 + 4 * j + c);
        sv = s ? __ldg(reinterpret_cast<const float4*>(s + gg * kGroup) + lane)
               : make_float4(1.f, 1.f, 1.f, 1.f);
    };
    bool bad = false;
    uint4 raw[4];
    float4 sv;
    if (unit0 < units) fetch(chunk, g, raw, sv);
    // every lane runs the same number of iterations (the shuffles and votes
    // need the whole warp); lanes past the last row work on row N - 1 and
    // write nothing.  The next unit's loads are issued before this unit's
    // arithmetic.
    for (int64_t u = unit0; u < units; u += stride) {
        const int64_t n = chunk * 8 + rg;
        const bool live = n < N;
        const int64_t nn = live ? n : N - 1;
        int64_t g_next = g + sr, chunk_next = chunk + sq;
        if (g_next >= G) {
            g_next -= G;
            ++chunk_next;
        }
        uint4 raw_next[4];
        float4 sv_next;
        if (u + stride < units) fetch(chunk_next, g_next, raw_next, sv_next);   // warp-uniform
        __syncwarp();                       // the previous unit's reads of ss are done
        reinterpret_cast<float4*>(ss)[lane] = sv;
        __syncwarp();
        float2 wp2[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 sa = reinterpret_cast<const float4*>(ss)[8 * j + 2 * c];
            const float4 sb = reinterpret_cast<const float4*>(ss)[8 * j + 2 * c + 1];
            const float2 sf[4] = {make_float2(sa.x, sa.y), make_float2(sa.z, sa.w),
                                  make_float2(sb.x, sb.y), make_float2(sb.z, sb.w)};
            const uint32_t rw[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                wp2[4 * j + h] =
                    __fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&rw[h])), sf[h]);
        }
        // four independent min / max chains, then their combination
        float lq[4], hq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            lq[q] = fmin_nan(wp2[q].x, wp2[q].y);
            hq[q] = fmax_nan(wp2[q].x, wp2[q].y);
        }
#pragma unroll
        for (int e = 4; e < 16; ++e) {
            lq[e & 3] = fmin3_nan(lq[e & 3], wp2[e].x, wp2[e].y);
            hq[e & 3] = fmax3_nan(hq[e & 3], wp2[e].x, wp2[e].y);
        }
        float lo = fmin_nan(fmin3_nan(lq[0], lq[1], lq[2]), lq[3]);
        float hi = fmax_nan(fmax3_nan(hq[0], hq[1], hq[2]), hq[3]);
        const float* wp = reinterpret_cast<const float*>(wp2);
        // this lane's 32 values: NaN or Inf makes lo or hi non-finite
        const bool lane_bad = !(isfinite(lo) && isfinite(hi));
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        const GroupQuant gq = group_quant_from_range(lo, hi, kQmax);
        if (live) bad |= lane_bad || !gq.finite;
        const bool inside = rint_small(__fmul_rn(lo, gq.rcp)) >= -gq.zf &&
                            rint_small(__fmul_rn(hi, gq.rcp)) <= kQmax - gq.zf;
        uint32_t w[4];
        const bool tie = __all_sync(0xffffffffu, inside)
                             ? fast_nibbles32<false>(wp2, gq.rcp, gq.zf, kQmax, w)
                             : fast_nibbles32<true>(wp2, gq.rcp, gq.zf, kQmax, w);
        if (__any_sync(0xffffffffu, tie)) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = nibbles8_exact(wp + 8 * i, gq.scale, gq.rcp, gq.zf, kQmax);
        }
        if constexpr (BITS == 4) {
            if (live) {
                uint32_t* pw = out + nn * (K / 8) + g * 16 + c;
#pragma unroll
                for (int j = 0; j < 4; ++j) pw[4 * j] = w[j];
            }
        } else {
            uint32_t pl[3];
#pragma unroll
            for (int p = 0; p < 3; ++p) {
                uint32_t v = nibble_plane(w[0], p) | (nibble_plane(w[1], p) << 8) |
                             (nibble_plane(w[2], p) << 16) | (nibble_plane(w[3], p) << 24);
                v = __byte_perm(v, __shfl_xor_sync(0xffffffffu, v, 2), sel2);
                pl[p] = __byte_perm(v, __shfl_xor_sync(0xffffffffu, v, 1), sel1);
            }
            if (live) {
                uint32_t* pw = out + nn * (K / 32 * 3) + g * 12 + 3 * c;
#pragma unroll
                for (int p = 0; p < 3; ++p) pw[p] = pl[p];
            }
        }
        if (live && c == 0) {
            scales[nn * G + g] = __half_as_ushort(gq.scale_h);
            zeros[nn * G + g] = __half_as_ushort(__float2half_rn(gq.zf));
        }
        g = g_next;
        chunk = chunk_next;
#pragma unroll
        for (int j = 0; j < 4; ++j) raw[j] = raw_next[j];
        sv = sv_next;
    }
    if (bad) set_status(status, kStatusNonFinite);
}

// mse[a] = (sum of alpha a's partials) / (T N): one warp per alpha, lane-
// strided fp64 sums added in a fixed butterfly order (deterministic); then
// the first argmin and its candidate scales.
__global__ void __launch_bounds__(1024)
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
        // loads of 8 strides in flight at a time; the adds stay in order
#pragma unroll 8
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

// inv[i] = fp32(1 / s[i]) correctly rounded (the candidate kernel's rule).
__global__ void __launch_bounds__(256)
    reciprocal_kernel(const float* __restrict__ s, int64_t n, float* __restrict__ inv) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        inv[i] = __frcp_rn(s[i]);
}

// Xs = fp16(fp32(X) * inv_s), 8 activations per thread (K % 8 == 0).
__global__ void __launch_bounds__(256)
    scale_x_kernel(const uint16_t* __restrict__ X, int64_t M, int64_t K, int64_t ldx,
                   const float* __restrict__ inv_s, uint16_t* __restrict__ Xs) {
    grid_dep_launch();          // the matmul's set-up and weight loads may start now
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

// A warp per unit of eight rows of one group, at most kPackBlocksPerSm
// blocks per SM.
unsigned pack_blocks(int64_t N, int64_t K, int num_sms) {
    const int64_t units = (N + 7) / 8 * (K / kGroup);
    const int64_t warps = kPackThreads / 32;
    const int64_t blocks = (units + warps - 1) / warps;
    const int64_t cap = (int64_t)num_sms * kPackBlocksPerSm;
    return (unsigned)(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_reciprocals(const float* s, int64_t n, float* inv, int num_sms,
                               cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    reciprocal_kernel<<<(unsigned)blocks, 256, 0, st>>>(s, n, inv);
    return cudaGetLastError();
}

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
    const dim3 grid(cand_blocks(K), n_alpha);
    cand_pass1_kernel<<<grid, kCandThreads, 0, st>>>(mean, K, alphas, ws_r, ws_mm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const dim3 grid2((unsigned)((K + kCand2Threads - 1) / kCand2Threads), n_alpha);
    cand_pass2_kernel<<<grid2, kCand2Threads, 0, st>>>(K, cand_blocks(K), ws_r, ws_mm, s_alpha,
                                                      inv_s_alpha);
    return cudaGetLastError();
}

cudaError_t launch_pack_int4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                             uint32_t* qweight, uint16_t* scales, uint16_t* zeros, unsigned* status,
                             int num_sms, cudaStream_t st) {
    const int64_t items = N * (K / kGroup);
    if (items == 0) return cudaSuccess;
    pack_kernel<4><<<pack_blocks(N, K, num_sms), kPackThreads, 0, st>>>(W, N, K, ldw, s, qweight, scales,
                                                                 zeros, status);
    return cudaGetLastError();
}

cudaError_t launch_pack_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                             uint32_t* planes, uint16_t* scales, uint16_t* zeros, unsigned* status,
                             int num_sms, cudaStream_t st) {
    const int64_t items = N * (K / kGroup);
    if (items == 0) return cudaSuccess;
    pack_kernel<3><<<pack_blocks(N, K, num_sms), kPackThreads, 0, st>>>(W, N, K, ldw, s, planes, scales,
                                                                 zeros, status);
    return cudaGetLastError();
}

cudaError_t launch_search_finalize(const double* partials, int n_alpha, int64_t n_part, int64_t T,
                                   int64_t N, int64_t K, const float* s_alpha, double* mse,
                                   int32_t* best_idx, float* s_out, cudaStream_t st) {
    // one warp per alpha (AWQ_MAX_ALPHAS = 64 at most, 32 warps: two rounds)
    search_finalize_kernel<<<1, 1024, 0, st>>>(partials, n_alpha, n_part, T, N, K, s_alpha, mse,
                                               best_idx, s_out);
    return cudaGetLastError();
}

}  // namespace awq
