// W4A16 decode matmul for M <= 16 tokens: Y[M,N] = X[M,K] deq(Wq)^T.
//
// Decoding reads every weight once per step and does little arithmetic with
// it ("AWQ: Activation-aware Weight Quantization ...", fdeinterviews.com/
// papers/awq, first paragraph), so this kernel exists to stream the packed
// words at HBM speed:
//
//  * Persistent grid, one CTA per SM.  CTA c owns a balanced, contiguous run
//    of 16-row slabs; its consumer warps (16 for up to 8 tokens, else 8)
//    split the CTA's (slab, 5-group chunk) units into equal contiguous
//    ranges, so a slab can be shared by neighbouring warps (intra-CTA
//    split-K).
//  * Each warp streams its units through its own ring in shared memory,
//    filled by TMA: one 2-D box of 16 rows x 5 groups (320 contiguous bytes
//    per row) per unit.  With a 320-byte row pitch the fragment reads of a
//    quarter warp (two rows, 4 x 16 B each) fall on disjoint bank halves.
//    Narrow boxes (one 64-byte group per row) are not used: on B300 the TMA
//    then issues one small request per row and delivers only about 1 TB/s.
//    Every warp's whole ring is requested at kernel start: 160 KB per SM in
//    flight.
//  * Nibbles become exact fp16 values (q - z) in registers: a LOP3 places a
//    nibble in the mantissa of 1024.0 (or 1024 + 16 q for the high nibble of
//    a byte), and one HSUB2 / HFMA2 removes the offset and the zero-point.
//    (q - z) is an integer in [-15, 15], so nothing is rounded.
//  * The products go to the tensor cores through register-sourced
//    mma.m16n8k16 (fp16 in, fp32 accumulate), which keeps the M FMAs per
//    weight off the FP32 pipe.  The MMA's k order is a permutation of the
//    physical k order chosen so that each thread's 16 loaded bytes of a row
//    are exactly its A fragment; each thread reads the matching 64 bytes of
//    activations (L1-resident) and applies the same permutation with PRMT.
//    The group scale is applied in fp32 to the per-group partial sums.
//  * A slab owned by one warp is written straight from registers; a slab
//    shared by several warps is reduced through shared memory in warp order.
//    The work split depends on N and K only, so the result is deterministic
//    and independent of M, and the kernel needs no workspace.
#include "common.cuh"
#include "kernels.cuh"

namespace awq {
namespace {

constexpr int kDecRows = 16;                        // rows per slab (MMA M)
// Groups per ring stage.  One TMA box per stage: 16 rows x kDecChunk groups
// (row pitch kDecChunk * 64 B in shared memory).  An odd count makes the
// pitch an odd multiple of 64 B, so the two rows a quarter warp reads sit on
// disjoint bank halves; wide rows keep the TMA's per-row request count low.
constexpr int kDecChunk = 5;
constexpr int kDecPitch = kDecChunk * 64;                     // 320 B
constexpr int kDecStageBytes = kDecRows * kDecPitch;          // 5 KB
static_assert(kDecChunk % 2 == 1, "row pitch must be an odd multiple of 64 bytes");

// Consumer warps per CTA: 16 with a 2-stage ring each for up to 8 tokens,
// 8 (more registers each) with a 3-stage ring for 9..16 tokens.
template <int NW>
struct DecCfg {
    static constexpr int kThreads = NW * 32;
    static constexpr int kStages = NW >= 16 ? 2 : 3;
    static constexpr int kSlots = 2 * NW;           // partial sums: first/last slab of each warp
    static constexpr size_t kRingBytes = (size_t)NW * kStages * kDecStageBytes;
    static constexpr size_t kPartBytes = (size_t)kSlots * kDecRows * 16 * sizeof(float);
    static constexpr size_t kCtlBytes = (size_t)NW * kStages * 8 + (size_t)NW * 12 + 16;
    static constexpr size_t kSmem = 1024 + kRingBytes + kPartBytes + kCtlBytes;
};
static_assert(DecCfg<16>::kSmem <= 232448 && DecCfg<8>::kSmem <= 232448,
              "decode kernel exceeds shared memory");

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

// Per-group operands a thread needs besides the weights: the scale and
// zero-point of its two rows, and its 64 bytes of each token's activations.
template <int NB>
struct GroupIn {
    uint16_t sa, sb, za, zb;
    uint4 x[NB][4];
};

template <int NB>
__device__ __forceinline__ void load_group_in(GroupIn<NB>& in, const GemvParams& p, int64_t row_a,
                                              int gi, int g, int t) {
    const bool va = row_a < p.N, vb = row_a + 8 < p.N;
    in.sa = va ? __ldg(p.scales + row_a * p.G + gi) : (uint16_t)0;
    in.za = va ? __ldg(p.zeros + row_a * p.G + gi) : (uint16_t)0;
    in.sb = vb ? __ldg(p.scales + (row_a + 8) * p.G + gi) : (uint16_t)0;
    in.zb = vb ? __ldg(p.zeros + (row_a + 8) * p.G + gi) : (uint16_t)0;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int tok = g + 8 * nb;
        if (tok < p.M) {
            const uint4* xp = reinterpret_cast<const uint4*>(p.X + (int64_t)tok * p.ldx +
                                                             (int64_t)gi * kGroup + 32 * t);
#pragma unroll
            for (int i = 0; i < 4; ++i) in.x[nb][i] = __ldg(xp + i);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) in.x[nb][i] = make_uint4(0, 0, 0, 0);
        }
    }
}

// y += scale * (X_group (q - z)^T) for one group: 8 (16 for NB = 2) MMAs in
// four independent accumulator chains (one per packed word), added in a
// fixed order.
template <int NB>
__device__ __forceinline__ void group_mma(float (&y)[NB][4], const GroupIn<NB>& in, uint4 wa,
                                          uint4 wb) {
    const __half za = __ushort_as_half(in.za), zb = __ushort_as_half(in.zb);
    const __half h1024 = __float2half_rn(1024.0f), h64 = __float2half_rn(64.0f);
    const __half2 za1024 = __half2half2(__hadd(h1024, za));
    const __half2 zb1024 = __half2half2(__hadd(h1024, zb));
    const __half2 zaneg = __half2half2(__hneg(__hadd(h64, za)));
    const __half2 zbneg = __half2half2(__hneg(__hadd(h64, zb)));
    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
    float c[NB][4][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) c[nb][i][j] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t pa[4], pb[4];
        dequant_word(wA[i], za1024, zaneg, pa);
        dequant_word(wB[i], zb1024, zbneg, pb);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const uint4 b = permute_x8(in.x[nb][i]);
            mma16816(c[nb][i], pa[0], pb[0], pa[1], pb[1], b.x, b.y);
            mma16816(c[nb][i], pa[2], pb[2], pa[3], pb[3], b.z, b.w);
        }
    }
    const float fsa = __half2float(__ushort_as_half(in.sa));
    const float fsb = __half2float(__ushort_as_half(in.sb));
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        float s[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            s[j] = (c[nb][0][j] + c[nb][1][j]) + (c[nb][2][j] + c[nb][3][j]);
        y[nb][0] = fmaf(fsa, s[0], y[nb][0]);
        y[nb][1] = fmaf(fsa, s[1], y[nb][1]);
        y[nb][2] = fmaf(fsb, s[2], y[nb][2]);
        y[nb][3] = fmaf(fsb, s[3], y[nb][3]);
    }
}

// First unit of warp j when U units are split over NW warps (NW a power of
// two, so the division is a shift).
template <int NW>
__device__ __forceinline__ int warp_lo(int U, int j) {
    return (int)(((int64_t)j * U) / NW);
}

template <int NW>
struct DecCtl {
    uint64_t full[NW][DecCfg<NW>::kStages];
    int w_lo[NW], w_hi[NW], w_first[NW];    // each warp's unit range and first slab
    int abort;
};
static_assert(sizeof(DecCtl<16>) <= DecCfg<16>::kCtlBytes &&
                  sizeof(DecCtl<8>) <= DecCfg<8>::kCtlBytes,
              "control block does not fit its shared-memory slot");

template <int NB, int NW>
__global__ void __launch_bounds__(NW * 32, 1)
    gemv_w4a16_kernel(const __grid_constant__ CUtensorMap mapW, const GemvParams p) {
    using Cfg = DecCfg<NW>;
    constexpr int kDecWarps = NW;
    constexpr int kDecThreads = Cfg::kThreads;
    constexpr int kDecStages = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ring = smem;
    float* part = reinterpret_cast<float*>(smem + Cfg::kRingBytes);
    DecCtl<NW>* ctl = reinterpret_cast<DecCtl<NW>*>(smem + Cfg::kRingBytes + Cfg::kPartBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;

    // ---- work split: slabs over CTAs, (slab, chunk) units over warps ----
    // CTA-local unit indices fit in 32 bits (checked on the host), and the
    // loop walks (slab, chunk) incrementally: no 64-bit division anywhere.
    const int n_slabs = (int)((p.N + kDecRows - 1) / kDecRows);
    const int CG = (p.G + kDecChunk - 1) / kDecChunk;
    const int s0 = (int)((int64_t)blockIdx.x * n_slabs / gridDim.x);
    const int s1 = (int)((int64_t)(blockIdx.x + 1) * n_slabs / gridDim.x);
    const int U = (s1 - s0) * CG;
    const int u_lo = warp_lo<NW>(U, warp), u_hi = warp_lo<NW>(U, warp + 1);
    const int n_my = u_hi - u_lo;
    const int first_sl = u_lo / CG;                     // this warp's first CTA-local slab
    uint8_t* my_ring = ring + (size_t)warp * kDecStages * kDecStageBytes;

    if (lane == 0) {
        for (int s = 0; s < kDecStages; ++s) mbar_init(&ctl->full[warp][s], 1);
        fence_mbar_init();
        ctl->w_lo[warp] = u_lo;
        ctl->w_hi[warp] = u_hi;
        ctl->w_first[warp] = first_sl;
    }
    if (threadIdx.x == 0) {
        ctl->abort = 0;
        tma_prefetch_desc(&mapW);
    }
    __syncthreads();

    // lane 0: request unit u (CTA-local) into ring stage s: one box of 16
    // rows x kDecChunk groups (groups past K and rows past N are zero-filled
    // and still count toward the box's bytes)
    auto issue = [&](int u, int s) {
        const int sl = u / CG;
        const int ch = u - sl * CG;
        uint64_t* bar = &ctl->full[warp][s];
        mbar_arrive_expect_tx(bar, (uint32_t)kDecStageBytes);
        tma_load_2d(my_ring + (size_t)s * kDecStageBytes, &mapW, bar, ch * kDecChunk * 16,
                    (s0 + sl) * kDecRows);
    };
    if (lane == 0)
        for (int i = 0; i < kDecStages && i < n_my; ++i) issue(u_lo + i, i);
    __syncwarp();

    // write a finished slab: straight to Y when this warp owns the whole
    // slab, else into this warp's first/last partial slot
    auto flush = [&](int sl, const float (&y)[NB][4]) {
        const bool owned = sl * CG >= u_lo && (sl + 1) * CG <= u_hi;
        const int64_t row0 = (int64_t)(s0 + sl) * kDecRows;
        if (owned) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tok = nb * 8 + 2 * t + (j & 1);
                    const int64_t row = row0 + g + ((j < 2) ? 0 : 8);
                    if (tok < p.M && row < p.N)
                        p.Y[(int64_t)tok * p.ldy + row] =
                            __half_as_ushort(__float2half_rn(y[nb][j]));
                }
        } else {
            const int slot = 2 * warp + (sl == first_sl ? 0 : 1);
            float* dst = part + (size_t)slot * kDecRows * 16;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tok = nb * 8 + 2 * t + (j & 1);
                    const int rl = g + ((j < 2) ? 0 : 8);
                    dst[rl * 16 + tok] = y[nb][j];
                }
        }
    };

    float y[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int j = 0; j < 4; ++j) y[nb][j] = 0.0f;
    int cur = -1;
    int sl = first_sl, ch = u_lo - first_sl * CG;       // (slab, chunk) of unit u_lo + i
    int i = 0;
    bool ok = true;
    for (; i < n_my; ++i) {
        if (sl != cur) {
            if (cur >= 0) flush(cur, y);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int j = 0; j < 4; ++j) y[nb][j] = 0.0f;
            cur = sl;
        }
        const int64_t row_a = (int64_t)(s0 + sl) * kDecRows + g;
        const int gb = ch * kDecChunk, ge = min(p.G, gb + kDecChunk);
        // operands of the chunk's first group go out before the wait
        GroupIn<NB> nxt;
        load_group_in<NB>(nxt, p, row_a, gb, g, t);
        const int s = i % kDecStages;
        if (!mbar_wait(&ctl->full[warp][s], (uint32_t)(i / kDecStages) & 1u, &ctl->abort,
                       p.status)) {
            ok = false;
            break;
        }
        const uint8_t* box = my_ring + (size_t)s * kDecStageBytes;
#pragma unroll
        for (int jg = 0; jg < kDecChunk; ++jg) {
            const int gi = gb + jg;
            if (gi < ge) {
                const GroupIn<NB> in = nxt;
                if (gi + 1 < ge) load_group_in<NB>(nxt, p, row_a, gi + 1, g, t);
                const uint8_t* gbox = box + jg * 64 + t * 16;
                const uint4 wa = *reinterpret_cast<const uint4*>(gbox + g * kDecPitch);
                const uint4 wb = *reinterpret_cast<const uint4*>(gbox + (g + 8) * kDecPitch);
                group_mma<NB>(y, in, wa, wb);
            }
        }
        __syncwarp();
        if (lane == 0 && i + kDecStages < n_my) {
            // the warp's reads of this stage are done; TMA may overwrite it
            fence_proxy_async_smem();
            issue(u_lo + i + kDecStages, s);
        }
        if (++ch == CG) {
            ch = 0;
            ++sl;
        }
    }
    if (ok && cur >= 0) flush(cur, y);
    if (!ok && lane == 0) {
        // bounded drain of the copies this warp still has in flight
        for (int k = i; k < n_my && k < i + kDecStages; ++k) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&ctl->full[warp][k % kDecStages], (uint32_t)(k / kDecStages) & 1u))
                if (globaltimer_ns() - t0 > 100000000ull) break;
        }
    }
    __syncthreads();
    if (ctl->abort) return;

    // ---- slabs shared by several warps: add the partials in warp order ----
    // The slab holding warp b's first unit is shared when that unit is not
    // the slab's first; the lowest such b reduces it, all such slabs at once.
    if (warp >= 1 && u_lo < U && u_lo % CG != 0) {
        const int rsl = u_lo / CG;
        if (ctl->w_lo[warp - 1] <= rsl * CG) {
            const int64_t row0 = (int64_t)(s0 + rsl) * kDecRows;
            for (int e = lane; e < kDecRows * p.M; e += 32) {
                const int r = e / p.M, m = e - r * p.M;
                float acc = 0.0f;
                for (int j = 0; j < NW; ++j) {
                    const int lo = ctl->w_lo[j], hi = ctl->w_hi[j];
                    if (hi <= lo || hi <= rsl * CG || lo >= (rsl + 1) * CG) continue;
                    const int slot = 2 * j + (ctl->w_first[j] == rsl ? 0 : 1);
                    acc += part[(slot * kDecRows + r) * 16 + m];
                }
                const int64_t row = row0 + r;
                if (row < p.N)
                    p.Y[(int64_t)m * p.ldy + row] = __half_as_ushort(__float2half_rn(acc));
            }
        }
    }
}

template <int NB, int NW>
cudaError_t launch_gemv_nb(const CUtensorMap& mapW, const GemvParams& p, int grid,
                           cudaStream_t st) {
    constexpr size_t smem = DecCfg<NW>::kSmem;
    cudaError_t e = smem_attr_once<gemv_w4a16_kernel<NB, NW>>((int)smem);
    if (e != cudaSuccess) return e;
    gemv_w4a16_kernel<NB, NW><<<grid, DecCfg<NW>::kThreads, smem, st>>>(mapW, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const CUtensorMap& mapW, const GemvParams& p, int num_sms,
                        cudaStream_t st) {
    if (p.M <= 0 || p.N <= 0) return cudaSuccess;
    const int64_t n_slabs = (p.N + kDecRows - 1) / kDecRows;
    const int grid = (int)(n_slabs < num_sms ? n_slabs : num_sms);
    // the kernel indexes a CTA's (slab, chunk) units in 32 bits
    const int64_t cg = (p.G + kDecChunk - 1) / kDecChunk;
    if ((n_slabs / grid + 1) * cg * 16 >= (1LL << 31)) return cudaErrorInvalidValue;
    return p.M <= 8 ? launch_gemv_nb<1, 16>(mapW, p, grid, st)
                    : launch_gemv_nb<2, 8>(mapW, p, grid, st);
}

}  // namespace awq
