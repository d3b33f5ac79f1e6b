// Device helpers of the W4A16 decode kernels (M <= 16 tokens), shared by the
// kernel over the plain packed layout (gemv.cu) and the kernel over the
// repacked decode tiles (gemv_tiles.cu):
//  * nibbles become exact fp16 values (q - z) in registers: a LOP3 places a
//    nibble in the mantissa of 1024.0 (or 1024 + 16 q for the high nibble of
//    a byte), and one HSUB2 / HFMA2 removes the offset and the zero-point;
//  * the products go to the tensor cores through register-sourced
//    mma.m16n8k16 (fp16 in, fp32 accumulate).  A thread's four consecutive
//    packed words of a row (16 bytes, 32 physical k) are exactly its A
//    fragments of two MMAs under a fixed permutation of k, and the
//    activations are staged (or loaded) under the same permutation;
//  * the group scale is applied in fp32 to each group's partial sums.
#pragma once

#include "common.cuh"

namespace awq {
namespace dec {

constexpr int kDecRows = 16;                        // rows per slab (MMA M)

// Shared-memory activations: per token a row of G * 256 + 64 bytes; within
// a group, the 8-element chunk of physical k = 32 t + 8 i sits at chunk
// position 4 i + t already in fragment order (x0,x4)(x1,x5)(x2,x6)(x3,x7).
// The 64-byte pad puts consecutive tokens on different bank halves.
__host__ __device__ constexpr int64_t dec_x_row_bytes(int64_t G) { return G * 256 + 64; }

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// One 32-bit word (8 nibbles n0..n7, n_i at bits 4i) -> four fp16x2 pairs
// (n0,n4) (n1,n5) (n2,n6) (n3,n7), each minus the zero-point, exact.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 z1024, __half2 zneg64,
                                             uint32_t (&p)[4]) {
    const uint32_t magic = 0x64006400u;               // fp16x2 (1024, 1024)
    const __half2 sixteenth = __half2half2(__float2half_rn(0.0625f));
    uint32_t v0 = lop3_and_or(w, 0x000F000Fu, magic);        // 1024 + n0 | 1024 + n4
    uint32_t v1 = lop3_and_or(w, 0x00F000F0u, magic);        // 1024 + 16 n1 | ...
    uint32_t w8 = w >> 8;
    uint32_t v2 = lop3_and_or(w8, 0x000F000Fu, magic);       // n2 | n6
    uint32_t v3 = lop3_and_or(w8, 0x00F000F0u, magic);       // 16 n3 | 16 n7
    p[0] = h2_as_u32(__hsub2(u32_as_h2(v0), z1024));
    p[1] = h2_as_u32(__hfma2(u32_as_h2(v1), sixteenth, zneg64));
    p[2] = h2_as_u32(__hsub2(u32_as_h2(v2), z1024));
    p[3] = h2_as_u32(__hfma2(u32_as_h2(v3), sixteenth, zneg64));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// x * inv_s for 8 consecutive activations: fp32 product, rounded once to
// fp32 and once to fp16 (the fused form of the caller's "divide by s").
__device__ __forceinline__ uint4 scale_x8(uint4 v, const float* inv_s) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(inv_s));
    const float4 b = __ldg(reinterpret_cast<const float4*>(inv_s) + 1);
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
        const __half2 r = __floats2half2_rn(__fmul_rn(__low2float(h), f[2 * j]),
                                            __fmul_rn(__high2float(h), f[2 * j + 1]));
        w[j] = *reinterpret_cast<const uint32_t*>(&r);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// 8 physical activations (x0..x7) -> the B-fragment order of the permuted k:
// (x0,x4) (x1,x5) (x2,x6) (x3,x7).
__device__ __forceinline__ uint4 permute_x8(uint4 v) {
    uint4 o;
    o.x = prmt(v.x, v.z, 0x5410);
    o.y = prmt(v.x, v.z, 0x7632);
    o.z = prmt(v.y, v.w, 0x5410);
    o.w = prmt(v.y, v.w, 0x7632);
    return o;
}

// A thread's 64 bytes of each token's activations for one group, in
// fragment order (used when the activations are not staged in shared memory).
template <int NB>
struct GroupX {
    uint4 x[NB][4];
};

template <int NB>
__device__ __forceinline__ void load_group_x(GroupX<NB>& in, const uint16_t* X, int64_t ldx, int M,
                                             const float* inv_s, int gi, int g, int t) {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        // lanes of absent tokens read the last token (their column is dropped)
        const int tok = min(g + 8 * nb, M - 1);
        const uint4* xp = reinterpret_cast<const uint4*>(X + (int64_t)tok * ldx +
                                                         (int64_t)gi * kGroup + 32 * t);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 v = __ldg(xp + i);
            if (inv_s) v = scale_x8(v, inv_s + (int64_t)gi * kGroup + 32 * t + 8 * i);
            in.x[nb][i] = permute_x8(v);
        }
    }
}

// y += scale * (X_group (q - z)^T) for one group: 8 (16 for NB = 2) MMAs in
// two independent accumulator chains, added in a fixed order.  xs: this
// thread's staged activation rows (XS), one per n-tile, or null for a token
// beyond M.
template <int NB, bool XS>
__device__ __forceinline__ void group_mma(float (&y)[NB][4], uint16_t sa16, uint16_t sb16,
                                          uint16_t za16, uint16_t zb16, const GroupX<NB>& gx,
                                          uint4 wa, uint4 wb, const uint8_t* const (&xs)[NB],
                                          int gi, int t) {
    const __half za = __ushort_as_half(za16), zb = __ushort_as_half(zb16);
    const __half h1024 = __float2half_rn(1024.0f), h64 = __float2half_rn(64.0f);
    const __half2 za1024 = __half2half2(__hadd(h1024, za));
    const __half2 zb1024 = __half2half2(__hadd(h1024, zb));
    const __half2 zaneg = __half2half2(__hneg(__hadd(h64, za)));
    const __half2 zbneg = __half2half2(__hneg(__hadd(h64, zb)));
    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
    float c[NB][2][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) c[nb][i][j] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t pa[4], pb[4];
        dequant_word(wA[i], za1024, zaneg, pa);
        dequant_word(wB[i], zb1024, zbneg, pb);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            uint4 b;
            if constexpr (XS) {
                b = *reinterpret_cast<const uint4*>(xs[nb] + gi * 256 + (i * 4 + t) * 16);
            } else {
                b = gx.x[nb][i];
            }
            mma16816(c[nb][i & 1], pa[0], pb[0], pa[1], pb[1], b.x, b.y);
            mma16816(c[nb][i & 1], pa[2], pb[2], pa[3], pb[3], b.z, b.w);
        }
    }
    const float fsa = __half2float(__ushort_as_half(sa16));
    const float fsb = __half2float(__ushort_as_half(sb16));
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        y[nb][0] = fmaf(fsa, c[nb][0][0] + c[nb][1][0], y[nb][0]);
        y[nb][1] = fmaf(fsa, c[nb][0][1] + c[nb][1][1], y[nb][1]);
        y[nb][2] = fmaf(fsb, c[nb][0][2] + c[nb][1][2], y[nb][2]);
        y[nb][3] = fmaf(fsb, c[nb][0][3] + c[nb][1][3], y[nb][3]);
    }
}

// First unit of warp j when U units are split over NW warps (division by a
// compile-time constant).
template <int NW>
__device__ __forceinline__ int warp_lo(int U, int j) {
    return (int)(((int64_t)j * U) / NW);
}

// Stage the M x K activations in shared memory in fragment order (optionally
// scaled by inv_s): per token a row of dec_x_row_bytes(G) bytes; the chunk of
// physical k = 32 t + 8 i of group gl sits at gl * 256 + (4 i + t) * 16.
// Called by all nthreads threads of the block, followed by a barrier.
__device__ __forceinline__ void stage_x(uint8_t* xsm, const uint16_t* X, int64_t ldx, int M,
                                        const float* inv_s, int G, int tid, int nthreads) {
    const int64_t xrow = dec_x_row_bytes(G);
    const int chunks = M * G * 16;
    for (int cix = tid; cix < chunks; cix += nthreads) {
        const int m = cix / (G * 16), rem = cix - m * G * 16;
        const int gl = rem >> 4, k8 = rem & 15;
        uint4 v = __ldg(reinterpret_cast<const uint4*>(X + (int64_t)m * ldx +
                                                       (int64_t)gl * kGroup + k8 * 8));
        if (inv_s) v = scale_x8(v, inv_s + (int64_t)gl * kGroup + k8 * 8);
        const int tt = k8 >> 2, ii = k8 & 3;
        *reinterpret_cast<uint4*>(xsm + m * xrow + gl * 256 + (ii * 4 + tt) * 16) = permute_x8(v);
    }
}

// ---------------------------------------------------------------------------
// Folded zero-point (staged activations only).  With the magic-number
// conversion alone, an even nibble n of a word becomes the exact fp16 value
// 1024 + n and an odd one 1024 + 16 n.  Staging the activations as x' = x at
// even physical k and x' = x / 16 at odd k (a power-of-two scaling) makes
// every product x' v = 1024 x' + x q, so one group's MMA sum is
//   A = sum_k x'_k v_k = 1024 sum_k x'_k + sum_k x_k q_k,
// and its contribution to Y is scale * (A - (1024 sum x' + z sum x)).  The
// two per-(token, group) sums are formed once, in fp32, while staging; the
// dequantisation is then 4 LOP3 and 1 shift per 8 weights and nothing is
// subtracted per weight.  The 1024 sum x' term cancels against the same fp16
// x' values the MMA multiplied; what remains is fp32 rounding of sums about
// 10^3 times the per-group result, far below the fp16 output rounding.
// ---------------------------------------------------------------------------

// One word (8 nibbles n0..n7, n_i at bits 4i) -> the fp16x2 pairs
// (1024+n0, 1024+n4) (1024+16n1, 1024+16n5) (1024+n2, 1024+n6)
// (1024+16n3, 1024+16n7), exact.
__device__ __forceinline__ void dequant_word_biased(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t magic = 0x64006400u;               // fp16x2 (1024, 1024)
    p[0] = lop3_and_or(w, 0x000F000Fu, magic);
    p[1] = lop3_and_or(w, 0x00F000F0u, magic);
    const uint32_t w8 = w >> 8;
    p[2] = lop3_and_or(w8, 0x000F000Fu, magic);
    p[3] = lop3_and_or(w8, 0x00F000F0u, magic);
}

// d = A B with a zero accumulator (the first MMA of a chain).
__device__ __forceinline__ void mma16816_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Bytes of the per-(group, token) sums: for group gi, n-tile nb and lane
// column t, 16 bytes {1024 sum x', sum x} of tokens 8 nb + 2 t and
// 8 nb + 2 t + 1 (the two columns of that lane's C fragment).
__host__ __device__ constexpr int64_t dec_bs_bytes(int64_t G, int NB) { return G * NB * 64; }

// y += scale * (X'_group v^T - (1024 sum x' + z sum x)) for one group: 8
// (16 for NB = 2) MMAs in one chain per n-tile, from the staged x' rows
// (xs) and the staged sums (bs).  sz = {scale | zero << 16} of rows g and
// g + 8.
template <int NB>
__device__ __forceinline__ void group_mma_folded(float (&y)[NB][4], uint2 sz, uint4 wa, uint4 wb,
                                                 const uint8_t* const (&xs)[NB],
                                                 const uint8_t* bs, int gi, int t) {
    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
    float c[NB][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t pa[4], pb[4];
        dequant_word_biased(wA[i], pa);
        dequant_word_biased(wB[i], pb);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const uint4 b = *reinterpret_cast<const uint4*>(xs[nb] + gi * 256 + (i * 4 + t) * 16);
            if (i == 0)
                mma16816_zc(c[nb], pa[0], pb[0], pa[1], pb[1], b.x, b.y);
            else
                mma16816(c[nb], pa[0], pb[0], pa[1], pb[1], b.x, b.y);
            mma16816(c[nb], pa[2], pb[2], pa[3], pb[3], b.z, b.w);
        }
    }
    const float sa = __half2float(__ushort_as_half((unsigned short)(sz.x & 0xFFFFu)));
    const float za = __half2float(__ushort_as_half((unsigned short)(sz.x >> 16)));
    const float sb = __half2float(__ushort_as_half((unsigned short)(sz.y & 0xFFFFu)));
    const float zb = __half2float(__ushort_as_half((unsigned short)(sz.y >> 16)));
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const float4 q = *reinterpret_cast<const float4*>(bs + ((gi * NB + nb) * 4 + t) * 16);
        y[nb][0] = fmaf(sa, c[nb][0] - fmaf(za, q.y, q.x), y[nb][0]);
        y[nb][1] = fmaf(sa, c[nb][1] - fmaf(za, q.w, q.z), y[nb][1]);
        y[nb][2] = fmaf(sb, c[nb][2] - fmaf(zb, q.y, q.x), y[nb][2]);
        y[nb][3] = fmaf(sb, c[nb][3] - fmaf(zb, q.w, q.z), y[nb][3]);
    }
}

// stage_x for the folded route: x' (x, or x / 16 at odd k) in fragment order,
// and per (token, group) the fp32 sums {1024 sum x', sum x} into bs (layout
// of dec_bs_bytes).  The 16 chunks of one (token, group) are handled by the
// 16 lanes of a half-warp in the same pass (the chunk index advances by a
// multiple of 32), which add their sums in a fixed shuffle order.  Called by
// all nthreads threads (a multiple of 32), followed by a barrier.
template <int NB>
__device__ __forceinline__ void stage_x_folded(uint8_t* xsm, uint8_t* bs, const uint16_t* X,
                                               int64_t ldx, int M, const float* inv_s, int G,
                                               int tid, int nthreads) {
    const int64_t xrow = dec_x_row_bytes(G);
    const int chunks = M * G * 16;
    const int iters = (chunks + nthreads - 1) / nthreads;
    const __half2 sixteenth_odd = __halves2half2(__float2half_rn(1.0f), __float2half_rn(0.0625f));
    constexpr int kBatch = 4;                          // loads in flight per thread
    for (int it0 = 0; it0 < iters; it0 += kBatch) {
        uint4 v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int cix0 = tid + (it0 + b) * nthreads;
            const int cix = cix0 < chunks ? cix0 : chunks - 1;
            const int m = cix / (G * 16), rem = cix - m * G * 16;
            const int gl = rem >> 4, k8 = rem & 15;
            v[b] = __ldg(reinterpret_cast<const uint4*>(X + (int64_t)m * ldx +
                                                        (int64_t)gl * kGroup + k8 * 8));
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            if (it0 + b >= iters) break;              // uniform over the block
            const int cix0 = tid + (it0 + b) * nthreads;
            const bool live = cix0 < chunks;          // uniform over each half-warp
            const int cix = live ? cix0 : chunks - 1;
            const int m = cix / (G * 16), rem = cix - m * G * 16;
            const int gl = rem >> 4, k8 = rem & 15;
            uint4 x = v[b];
            if (inv_s) x = scale_x8(x, inv_s + (int64_t)gl * kGroup + k8 * 8);
            uint32_t w[4] = {x.x, x.y, x.z, x.w};
            float sx = 0.0f, sxp = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 h = u32_as_h2(w[j]);
                const __half2 hp = __hmul2(h, sixteenth_odd);   // (x_even, x_odd / 16)
                const float2 f = __half22float2(h), fp = __half22float2(hp);
                sx += f.x + f.y;
                sxp += fp.x + fp.y;
                w[j] = h2_as_u32(hp);
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                sx += __shfl_xor_sync(0xffffffffu, sx, o);
                sxp += __shfl_xor_sync(0xffffffffu, sxp, o);
            }
            if (live) {
                const int tt = k8 >> 2, ii = k8 & 3;
                *reinterpret_cast<uint4*>(xsm + m * xrow + gl * 256 + (ii * 4 + tt) * 16) =
                    permute_x8(make_uint4(w[0], w[1], w[2], w[3]));
                if (k8 == 0 && m < 8 * NB) {
                    const int nb = m >> 3, tcol = (m & 7) >> 1, slot = m & 1;
                    float* dst = reinterpret_cast<float*>(bs + ((gl * NB + nb) * 4 + tcol) * 16) +
                                 2 * slot;
                    dst[0] = 1024.0f * sxp;
                    dst[1] = sx;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 3-bit planes (three words per 32 levels: word p holds bit p of level i at
// bit i).  Rotating plane p right by (i - p) mod 32 puts bit i at bit p and
// bit i + 16 at bit 16 + p; OR-ing the three under the mantissa of fp16 1024
// gives the exact pair (1024 + q_i, 1024 + q_{i+16}), and an HSUB2 of
// (1024 + z) the exact pair (q_i - z, q_{i+16} - z).  Lane t of a row builds
// the pairs i = t, t + 4, t + 8, t + 12 of a block: its A fragments of two
// m16n8k16 MMAs, whose k order is a permutation of the block's levels; the
// activations are staged in the matching order (stage_x3).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t rotr32(uint32_t w, uint32_t n) { return __funnelshift_r(w, w, n); }

__device__ __forceinline__ uint32_t pair3_mz(uint32_t p0, uint32_t p1, uint32_t p2, uint32_t r0,
                                             uint32_t r1, uint32_t r2, __half2 z1024) {
    uint32_t v = lop3_and_or(rotr32(p0, r0), 0x00010001u, 0x64006400u);
    v = lop3_and_or(rotr32(p1, r1), 0x00020002u, v);
    v = lop3_and_or(rotr32(p2, r2), 0x00040004u, v);
    return h2_as_u32(__hsub2(u32_as_h2(v), z1024));
}

// Per token a row of K * 2 + 64 bytes; block j's 64 bytes hold, for lane
// column t = 0..3, the 16 bytes x[32 j + t + {0, 16, 4, 20, 8, 24, 12, 28}]
// (lane t's B fragments of the block's two MMAs).
__host__ __device__ constexpr int64_t dec_x3_row_bytes(int64_t K) { return K * 2 + 64; }

// Stage the M x K activations in that order: one thread per (token, block)
// loads the block's 64 bytes and writes its four 16-byte fragment groups.
// Called by all nthreads threads, followed by a barrier.
__device__ __forceinline__ void stage_x3(uint8_t* xsm, const uint16_t* X, int64_t ldx, int M,
                                         int64_t K, int tid, int nthreads) {
    const int64_t xrow = dec_x3_row_bytes(K);
    const int nblk = (int)(K / 32);
    for (int idx = tid; idx < M * nblk; idx += nthreads) {
        const int m = idx / nblk, j = idx - m * nblk;
        const uint4* src = reinterpret_cast<const uint4*>(X + (int64_t)m * ldx + 32 * (int64_t)j);
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldg(src + q);
            w[4 * q] = v.x;
            w[4 * q + 1] = v.y;
            w[4 * q + 2] = v.z;
            w[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            uint32_t o[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int lo = t + 4 * c, hi = lo + 16;     // levels of this pair
                const uint32_t sel = ((lo & 1) ? 0x3232u : 0x1010u) & 0x00FFu;
                const uint32_t selh = ((hi & 1) ? 0x7676u : 0x5454u) & 0xFF00u;
                o[c] = prmt(w[lo >> 1], w[hi >> 1], sel | selh);
            }
            *reinterpret_cast<uint4*>(xsm + (int64_t)m * xrow + (int64_t)j * 64 + t * 16) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// y += scale * (X_group (q - z)^T) for one group of the 3-bit tile rows g and
// g + 8 (plane words A and B, 12 each), 2 (4 for NB = 2) MMAs per 32-level
// block.  xs: the staged rows (XS), else the activations are read from X.
template <int NB, bool XS>
__device__ __forceinline__ void group_mma3(float (&y)[NB][4], uint2 sz, const uint32_t (&A)[12],
                                           const uint32_t (&B)[12], const uint8_t* const (&xs)[NB],
                                           const uint16_t* X, int64_t ldx, int M, int gi, int g,
                                           int t) {
    const __half h1024 = __float2half_rn(1024.0f);
    const __half2 za = __half2half2(__hadd(h1024, __ushort_as_half((unsigned short)(sz.x >> 16))));
    const __half2 zb = __half2half2(__hadd(h1024, __ushort_as_half((unsigned short)(sz.y >> 16))));
    float c[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int k = 0; k < 4; ++k) c[nb][k] = 0.0f;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t fa[4], fb[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const uint32_t r0 = (uint32_t)(t + 4 * cc) & 31u, r1 = (uint32_t)(t + 4 * cc - 1) & 31u,
                           r2 = (uint32_t)(t + 4 * cc - 2) & 31u;
            fa[cc] = pair3_mz(A[3 * blk], A[3 * blk + 1], A[3 * blk + 2], r0, r1, r2, za);
            fb[cc] = pair3_mz(B[3 * blk], B[3 * blk + 1], B[3 * blk + 2], r0, r1, r2, zb);
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            uint4 xb;
            if constexpr (XS) {
                xb = *reinterpret_cast<const uint4*>(xs[nb] + ((int64_t)gi * 4 + blk) * 64 + t * 16);
            } else {
                const int tok = min(g + 8 * nb, M - 1);
                const uint16_t* xp = X + (int64_t)tok * ldx + (int64_t)gi * kGroup + 32 * blk + t;
                uint32_t o[4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    o[cc] = (uint32_t)__ldg(xp + 4 * cc) | ((uint32_t)__ldg(xp + 4 * cc + 16) << 16);
                xb = make_uint4(o[0], o[1], o[2], o[3]);
            }
            mma16816(c[nb], fa[0], fb[0], fa[1], fb[1], xb.x, xb.y);
            mma16816(c[nb], fa[2], fb[2], fa[3], fb[3], xb.z, xb.w);
        }
    }
    const float sa = __half2float(__ushort_as_half((unsigned short)(sz.x & 0xFFFFu)));
    const float sb = __half2float(__ushort_as_half((unsigned short)(sz.y & 0xFFFFu)));
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        y[nb][0] = fmaf(sa, c[nb][0], y[nb][0]);
        y[nb][1] = fmaf(sa, c[nb][1], y[nb][1]);
        y[nb][2] = fmaf(sb, c[nb][2], y[nb][2]);
        y[nb][3] = fmaf(sb, c[nb][3], y[nb][3]);
    }
}

}  // namespace dec
}  // namespace awq
