// W4A16 decode matmul for M <= 16 tokens: Y[M,N] = X[M,K] deq(Wq)^T.
//
// Decoding reads every weight once per step and does little arithmetic with
// it ("AWQ: Activation-aware Weight Quantization ...", fdeinterviews.com/
// papers/awq, first paragraph), so this kernel is built to stream the packed
// words at HBM speed with the fewest instructions per weight:
//
//  * Each thread issues 128-bit loads of 32 consecutive nibbles (a quarter of
//    a group) of two weight rows; a warp covers 16 rows x one group of 128.
//  * Nibbles become exact fp16 values (q - z) in registers: a LOP3 places a
//    nibble in the mantissa of 1024.0 (or 1024 + 16 q for the high nibble of
//    a byte), and one HSUB2 / HFMA2 removes the offset and the zero-point.
//    (q - z) is an integer in [-15, 15], so nothing is rounded.
//  * The products go to the tensor cores through register-sourced
//    mma.m16n8k16 (fp16 in, fp32 accumulate), which keeps the M FMAs per
//    weight off the FP32 pipe: with CUDA-core FMAs alone the dequantise +
//    multiply work would cap the kernel below HBM speed.  Tensor memory and
//    shared-memory operands (tcgen05) would add an smem round trip per
//    weight, which costs more bandwidth than this path saves.
//  * The MMA's k order is a permutation of the physical k order chosen so
//    that each thread's loaded words are exactly its A-fragment; the
//    activations are staged in shared memory under the same permutation.
//    The group scale is applied in fp32 to the per-group partial sums.
//  * K is split over the CTAs of a thread-block cluster; partial sums are
//    reduced in a fixed order through distributed shared memory, so the
//    kernel needs no workspace and is deterministic.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.cuh"

namespace cg = cooperative_groups;

namespace awq {
namespace {

constexpr int kGemvWarps = 4;                 // 16 weight rows per warp
constexpr int kGemvRows = 16 * kGemvWarps;    // rows per CTA
constexpr int kGemvBatch = 4;                 // groups loaded ahead per warp
constexpr size_t kGemvSmemMax = 200 * 1024;

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

// Shared memory: the partial-sum tile [64 rows][M] fp32, then the
// activations of this CTA's K range, per token a row of ng*256 + 64 bytes
// (padding keeps the 16-byte fragment reads of a quarter warp on distinct
// banks).  Within a group the 8-element chunk of physical k = 32 t + 8 i is
// stored at chunk position 4 i + t, its elements in the order
// (0,4,1,5,2,6,3,7).
template <int NB>
__global__ void __launch_bounds__(kGemvWarps * 32)
    gemv_w4a16_kernel(GemvParams p, int cs) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x / cs, split = blockIdx.x % cs;
    const int gs = (int)((int64_t)split * p.G / cs), ge = (int)((int64_t)(split + 1) * p.G / cs);
    const int ng = ge - gs;
    const int M = p.M;
    const int64_t row_stride = (int64_t)ng * 256 + 64;   // bytes per token row
    // the partial-sum tile sits at offset 0 so that it has the same address
    // in every CTA of the cluster (their K ranges, hence xs sizes, differ)
    float* part = reinterpret_cast<float*>(smem);
    uint8_t* xs = smem + (size_t)kGemvRows * M * 4;

    // ---- stage X[:, gs*128 .. ge*128) with the fragment permutation ----
    const int chunks = M * ng * 16;
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        const int m = c / (ng * 16), rem = c - m * ng * 16;
        const int gl = rem >> 4, k8 = rem & 15;          // group, chunk within group
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(
            p.X + (int64_t)m * p.ldx + (int64_t)(gs + gl) * kGroup + k8 * 8));
        uint4 o;
        o.x = prmt(v.x, v.z, 0x5410);    // (x0, x4)
        o.y = prmt(v.x, v.z, 0x7632);    // (x1, x5)
        o.z = prmt(v.y, v.w, 0x5410);    // (x2, x6)
        o.w = prmt(v.y, v.w, 0x7632);    // (x3, x7)
        const int t = k8 >> 2, i = k8 & 3;
        *reinterpret_cast<uint4*>(xs + (int64_t)m * row_stride + gl * 256 + (i * 4 + t) * 16) = o;
    }
    __syncthreads();

    // ---- main loop: this warp's 16 rows over the CTA's groups ----
    const int g = lane >> 2, t = lane & 3;
    const int64_t n_base = (int64_t)rb * kGemvRows + warp * 16;
    const int64_t ra = n_base + g, rbw = n_base + g + 8;
    const bool va = ra < p.N, vb = rbw < p.N;
    const int64_t wstride = p.K / 8;     // words per row
    const uint32_t* qa = p.qw + (va ? ra : 0) * wstride + 4 * t;
    const uint32_t* qb = p.qw + (vb ? rbw : 0) * wstride + 4 * t;
    const uint16_t* sa_p = p.scales + (va ? ra : 0) * p.G;
    const uint16_t* sb_p = p.scales + (vb ? rbw : 0) * p.G;
    const uint16_t* za_p = p.zeros + (va ? ra : 0) * p.G;
    const uint16_t* zb_p = p.zeros + (vb ? rbw : 0) * p.G;
    // activation fragments: token columns g (and g + 8)
    const bool tok0 = g < M, tok1 = (NB == 2) && (g + 8 < M);
    const uint8_t* x0 = xs + (int64_t)(tok0 ? g : 0) * row_stride + t * 16;
    const uint8_t* x1 = xs + (int64_t)(tok1 ? g + 8 : 0) * row_stride + t * 16;

    float y[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int j = 0; j < 4; ++j) y[nb][j] = 0.0f;

    for (int gb = gs; gb < ge; gb += kGemvBatch) {
        uint4 wa[kGemvBatch], wb[kGemvBatch];
        uint16_t sca[kGemvBatch], scb[kGemvBatch], zea[kGemvBatch], zeb[kGemvBatch];
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u) {
            const int gi = gb + u;
            if (gi < ge) {
                wa[u] = va ? __ldg(reinterpret_cast<const uint4*>(qa + (int64_t)gi * 16))
                           : make_uint4(0, 0, 0, 0);
                wb[u] = vb ? __ldg(reinterpret_cast<const uint4*>(qb + (int64_t)gi * 16))
                           : make_uint4(0, 0, 0, 0);
                sca[u] = __ldg(sa_p + gi);
                scb[u] = __ldg(sb_p + gi);
                zea[u] = __ldg(za_p + gi);
                zeb[u] = __ldg(zb_p + gi);
            }
        }
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u) {
            const int gi = gb + u;
            if (gi >= ge) break;
            const __half za = __ushort_as_half(zea[u]), zb = __ushort_as_half(zeb[u]);
            const __half h1024 = __float2half_rn(1024.0f), h64 = __float2half_rn(64.0f);
            const __half2 za1024 = __half2half2(__hadd(h1024, za));
            const __half2 zb1024 = __half2half2(__hadd(h1024, zb));
            const __half2 zaneg = __half2half2(__hneg(__hadd(h64, za)));
            const __half2 zbneg = __half2half2(__hneg(__hadd(h64, zb)));
            const uint32_t wA[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
            const uint32_t wB[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
            const int64_t goff = (int64_t)(gi - gs) * 256;
            float c[NB][4];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int j = 0; j < 4; ++j) c[nb][j] = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t pa[4], pb[4];
                dequant_word(wA[i], za1024, zaneg, pa);
                dequant_word(wB[i], zb1024, zbneg, pb);
                uint4 b0 = tok0 ? *reinterpret_cast<const uint4*>(x0 + goff + i * 64)
                                : make_uint4(0, 0, 0, 0);
                mma16816(c[0], pa[0], pb[0], pa[1], pb[1], b0.x, b0.y);
                mma16816(c[0], pa[2], pb[2], pa[3], pb[3], b0.z, b0.w);
                if (NB == 2) {
                    uint4 b1 = tok1 ? *reinterpret_cast<const uint4*>(x1 + goff + i * 64)
                                    : make_uint4(0, 0, 0, 0);
                    mma16816(c[NB - 1], pa[0], pb[0], pa[1], pb[1], b1.x, b1.y);
                    mma16816(c[NB - 1], pa[2], pb[2], pa[3], pb[3], b1.z, b1.w);
                }
            }
            const float fsa = __half2float(__ushort_as_half(sca[u]));
            const float fsb = __half2float(__ushort_as_half(scb[u]));
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                y[nb][0] = fmaf(fsa, c[nb][0], y[nb][0]);
                y[nb][1] = fmaf(fsa, c[nb][1], y[nb][1]);
                y[nb][2] = fmaf(fsb, c[nb][2], y[nb][2]);
                y[nb][3] = fmaf(fsb, c[nb][3], y[nb][3]);
            }
        }
    }

    // ---- write out: C fragment = rows (g, g+8) x tokens (2t, 2t+1) (+8 nb) ----
    if (cs == 1) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tok = nb * 8 + 2 * t + (j & 1);
                const int64_t row = (j < 2) ? ra : rbw;
                if (tok < M && row < p.N)
                    p.Y[(int64_t)tok * p.ldy + row] = __half_as_ushort(__float2half_rn(y[nb][j]));
            }
        return;
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int tok = nb * 8 + 2 * t + (j & 1);
            const int rl = warp * 16 + g + ((j < 2) ? 0 : 8);
            if (tok < M) part[rl * M + tok] = y[nb][j];
        }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    // CTA `split` reduces its share of the [64 x M] tile over all ranks, in
    // rank order, and writes fp16.
    const int tile = kGemvRows * M;
    const int per = (tile + cs - 1) / cs;
    const int e0 = split * per, e1 = min(tile, e0 + per);
    for (int e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
        float acc = 0.0f;
        for (int q = 0; q < cs; ++q) acc += cluster.map_shared_rank(part, q)[e];
        const int rl = e / M, tok = e - rl * M;
        const int64_t row = (int64_t)rb * kGemvRows + rl;
        if (row < p.N) p.Y[(int64_t)tok * p.ldy + row] = __half_as_ushort(__float2half_rn(acc));
    }
    cluster.sync();
}

template <int NB>
cudaError_t launch_gemv_nb(const GemvParams& p, int num_sms, cudaStream_t st) {
    const int64_t n_rb = (p.N + kGemvRows - 1) / kGemvRows;
    auto smem_for = [&](int c) {
        const int max_ng = (p.G + c - 1) / c;
        return (size_t)p.M * ((size_t)max_ng * 256 + 64) + (size_t)kGemvRows * p.M * 4;
    };
    // split K over up to 8 CTAs: enough CTAs to fill the GPU, and few enough
    // groups per CTA for the staged activations to fit in shared memory
    int cs = 1;
    while (cs < 8 && 2 * cs <= p.G && (n_rb * cs < 4LL * num_sms || smem_for(cs) > kGemvSmemMax))
        cs *= 2;
    const size_t smem = smem_for(cs);
    if (smem > kGemvSmemMax) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemv_w4a16_kernel<NB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_rb * cs));
    cfg.blockDim = dim3(kGemvWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_w4a16_kernel<NB>, p, cs);
}

}  // namespace

cudaError_t launch_gemv(const GemvParams& p, int num_sms, cudaStream_t st) {
    if (p.M <= 0 || p.N <= 0) return cudaSuccess;
    return p.M <= 8 ? launch_gemv_nb<1>(p, num_sms, st) : launch_gemv_nb<2>(p, num_sms, st);
}

}  // namespace awq
