// W4A16 decode matmul for M <= 16 tokens: Y[M,N] = X[M,K] deq(Wq)^T.
//
// Decoding reads every weight once per step and does little arithmetic with
// it ("AWQ: Activation-aware Weight Quantization ...", fdeinterviews.com/
// papers/awq, first paragraph), so this kernel exists to stream the packed
// words at HBM speed:
//
//  * Persistent grid, one CTA per SM.  CTA c owns a balanced, contiguous run
//    of 16-row slabs; its consumer warps (16 for up to 8 tokens, else 8)
//    split the CTA's (slab, 3-group chunk) units into equal contiguous
//    ranges, so a slab can be shared by neighbouring warps (intra-CTA
//    split-K).
//  * Each warp streams its units through its own ring in shared memory,
//    filled by TMA: one 2-D box of 16 rows x 3 groups (192 contiguous bytes
//    per row) per unit.  With a 192-byte row pitch (an odd multiple of 64)
//    the fragment reads of a quarter warp (two rows, 4 x 16 B each) fall on
//    disjoint bank halves.  Every warp's whole ring is requested at kernel
//    start: 96 KB per SM in flight (16 warps x 2 stages x 3 KB).
//  * Nibbles become exact fp16 values (q - z) in registers: a LOP3 places a
//    nibble in the mantissa of 1024.0 (or 1024 + 16 q for the high nibble of
//    a byte), and one HSUB2 / HFMA2 removes the offset and the zero-point.
//    (q - z) is an integer in [-15, 15], so nothing is rounded.
//  * The products go to the tensor cores through register-sourced
//    mma.m16n8k16 (fp16 in, fp32 accumulate), which keeps the M FMAs per
//    weight off the FP32 pipe.  The MMA's k order is a permutation of the
//    physical k order chosen so that each thread's 16 loaded bytes of a row
//    are exactly its A fragment; the activations are staged once per CTA in
//    shared memory under the same permutation (or, when they do not fit,
//    read through L1 and permuted with PRMT).  The group scale is applied in
//    fp32 to the per-group partial sums.
//  * Programmatic dependent launch: the next kernel in the stream is released
//    at once and may take an SM as soon as this kernel's CTA there retires;
//    when the caller allows early weight reads it streams its first weights
//    before waiting for this kernel to complete.
//  * A slab owned by one warp is written straight from registers; a slab
//    shared by several warps is reduced through shared memory in warp order.
//    The work split depends on N and K only, so the result is deterministic
//    and independent of M, and the kernel needs no workspace.
#include "common.cuh"
#include "decode.cuh"
#include "kernels.cuh"

namespace awq {
namespace {

using namespace dec;
// Groups per ring stage.  One TMA box per stage: 16 rows x kDecChunk groups
// (row pitch kDecChunk * 64 B in shared memory).  An odd count makes the
// pitch an odd multiple of 64 B, so the two rows a quarter warp reads sit on
// disjoint bank halves; wide rows keep the TMA's per-row request count low.
constexpr int kDecChunk = 3;
constexpr int kDecPitch = kDecChunk * 64;                     // 192 B
constexpr int kDecStageBytes = kDecRows * kDecPitch;          // 3 KB
static_assert(kDecChunk % 2 == 1, "row pitch must be an odd multiple of 64 bytes");

// Per token-tile count NB (1: up to 8 tokens, 2: up to 16): 16 consumer
// warps with a 2-stage ring each for NB = 1, 8 warps (more registers each)
// with a 3-stage ring for NB = 2.  One CTA per SM.
template <int NB>
struct DecCfg {
    static constexpr int kWarps = NB == 1 ? 16 : 8;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kMinBlocks = 1;
    static constexpr int kStages = NB == 1 ? 2 : 3;
    static constexpr int kCols = 8 * NB;                // token columns (8 per MMA n-tile)
    static constexpr int kSlots = 2 * kWarps;           // partial sums: first/last slab of each warp
    static constexpr size_t kRingBytes = (size_t)kWarps * kStages * kDecStageBytes;
    static constexpr size_t kPartBytes = (size_t)kSlots * kDecRows * kCols * sizeof(float);
    static constexpr size_t kCtlBytes = (size_t)kWarps * 3 * 8 + (size_t)kWarps * 12 + 16;
    // fixed part; the staged activations (when they fit) follow it
    static constexpr size_t kSmem = 1024 + kRingBytes + kPartBytes + kCtlBytes;
};
constexpr size_t kDecSmemMax = 232448;                 // per-block opt-in limit on sm_103
static_assert(DecCfg<1>::kSmem <= kDecSmemMax && DecCfg<2>::kSmem <= kDecSmemMax,
              "decode kernel exceeds shared memory");

// Scale and zero-point of a thread's two rows for the groups of one chunk,
// loaded one chunk ahead.
struct ChunkSZ {
    uint16_t sa[kDecChunk], sb[kDecChunk], za[kDecChunk], zb[kDecChunk];
};

__device__ __forceinline__ void load_chunk_sz(ChunkSZ& z, const GemvParams& p, int64_t row_a,
                                              int gb) {
    const bool va = row_a < p.N, vb = row_a + 8 < p.N;
    const uint16_t* sa = p.scales + (va ? row_a : 0) * p.G;
    const uint16_t* za = p.zeros + (va ? row_a : 0) * p.G;
    const uint16_t* sb = p.scales + (vb ? row_a + 8 : 0) * p.G;
    const uint16_t* zb = p.zeros + (vb ? row_a + 8 : 0) * p.G;
#pragma unroll
    for (int j = 0; j < kDecChunk; ++j) {
        const int gi = gb + j;
        const bool in = gi < p.G;
        z.sa[j] = (va && in) ? __ldg(sa + gi) : (uint16_t)0;
        z.za[j] = (va && in) ? __ldg(za + gi) : (uint16_t)0;
        z.sb[j] = (vb && in) ? __ldg(sb + gi) : (uint16_t)0;
        z.zb[j] = (vb && in) ? __ldg(zb + gi) : (uint16_t)0;
    }
}

template <int NW>
struct DecCtl {
    uint64_t full[NW][3];
    int w_lo[NW], w_hi[NW], w_first[NW];    // each warp's unit range and first slab
    int abort;
};
static_assert(sizeof(DecCtl<16>) <= DecCfg<1>::kCtlBytes &&
                  sizeof(DecCtl<8>) <= DecCfg<2>::kCtlBytes && DecCfg<1>::kStages <= 3 &&
                  DecCfg<2>::kStages <= 3,
              "control block does not fit its shared-memory slot");

template <int NB, int NW, bool XS>
__global__ void __launch_bounds__(NW * 32, DecCfg<NB>::kMinBlocks)
    gemv_w4a16_kernel(const __grid_constant__ CUtensorMap mapW, const GemvParams p) {
    using Cfg = DecCfg<NB>;
    static_assert(Cfg::kWarps == NW, "warp count");
    constexpr int kDecThreads = Cfg::kThreads;
    constexpr int kDecStages = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ring = smem;
    float* part = reinterpret_cast<float*>(smem + Cfg::kRingBytes);
    DecCtl<NW>* ctl = reinterpret_cast<DecCtl<NW>*>(smem + Cfg::kRingBytes + Cfg::kPartBytes);
    uint8_t* xsm = smem + Cfg::kRingBytes + Cfg::kPartBytes + Cfg::kCtlBytes;   // XS only
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
    // Programmatic dependent launch: the next kernel in the stream may be
    // scheduled beside this one right away.  This kernel reads X and writes Y
    // only after griddepcontrol.wait, i.e. after the previous kernel has
    // completed and flushed; with early_weights (the caller's guarantee that
    // the previous kernel does not write the packed weights) the first ring
    // stages of weights are requested before that wait.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (p.early_weights && lane == 0)
        for (int i = 0; i < kDecStages && i < n_my; ++i) issue(u_lo + i, i);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!p.early_weights && lane == 0)
        for (int i = 0; i < kDecStages && i < n_my; ++i) issue(u_lo + i, i);
    __syncwarp();

    // stage the activations in fragment order while the first weights stream in
    const uint8_t* xs[NB];
    if constexpr (XS) {
        const int64_t xrow = dec_x_row_bytes(p.G);
        stage_x(xsm, p.X, p.ldx, p.M, p.inv_s, p.G, threadIdx.x, kDecThreads);
        __syncthreads();
        // an MMA output column depends only on its own B column, so lanes of
        // absent tokens read the last token's row and their outputs are dropped
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) xs[nb] = xsm + min(g + 8 * nb, p.M - 1) * xrow;
    } else {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) xs[nb] = nullptr;
    }

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
            float* dst = part + (size_t)slot * kDecRows * Cfg::kCols;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tok = nb * 8 + 2 * t + (j & 1);
                    const int rl = g + ((j < 2) ? 0 : 8);
                    dst[rl * Cfg::kCols + tok] = y[nb][j];
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
    ChunkSZ sz;
    if (n_my > 0) load_chunk_sz(sz, p, (int64_t)(s0 + sl) * kDecRows + g, ch * kDecChunk);
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
        const int gb = ch * kDecChunk, ge = min(p.G, gb + kDecChunk);
        // the next unit's scales and zero-points go out a chunk ahead
        int nsl = sl, nch = ch + 1;
        if (nch == CG) {
            nch = 0;
            ++nsl;
        }
        ChunkSZ nsz;
        if (i + 1 < n_my) load_chunk_sz(nsz, p, (int64_t)(s0 + nsl) * kDecRows + g, nch * kDecChunk);
        GroupX<NB> gx;
        if constexpr (!XS) load_group_x<NB>(gx, p.X, p.ldx, p.M, p.inv_s, gb, g, t);
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
                GroupX<NB> cx;
                if constexpr (!XS) {
                    cx = gx;
                    if (gi + 1 < ge) load_group_x<NB>(gx, p.X, p.ldx, p.M, p.inv_s, gi + 1, g, t);
                }
                const uint8_t* gbox = box + jg * 64 + t * 16;
                const uint4 wa = *reinterpret_cast<const uint4*>(gbox + g * kDecPitch);
                const uint4 wb = *reinterpret_cast<const uint4*>(gbox + (g + 8) * kDecPitch);
                group_mma<NB, XS>(y, sz.sa[jg], sz.sb[jg], sz.za[jg], sz.zb[jg], cx, wa, wb, xs,
                                  gi, t);
            }
        }
        __syncwarp();
        if (lane == 0 && i + kDecStages < n_my) {
            // the warp's reads of this stage are done; TMA may overwrite it
            fence_proxy_async_smem();
            issue(u_lo + i + kDecStages, s);
        }
        sz = nsz;
        sl = nsl;
        ch = nch;
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
                    acc += part[(slot * kDecRows + r) * Cfg::kCols + m];
                }
                const int64_t row = row0 + r;
                if (row < p.N)
                    p.Y[(int64_t)m * p.ldy + row] = __half_as_ushort(__float2half_rn(acc));
            }
        }
    }
}

template <int NB, int NW, bool XS>
cudaError_t launch_gemv_nb(const CUtensorMap& mapW, const GemvParams& p, int grid, size_t smem,
                           cudaStream_t st) {
    cudaError_t e = smem_attr_once<gemv_w4a16_kernel<NB, NW, XS>>((int)kDecSmemMax);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(DecCfg<NB>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_w4a16_kernel<NB, NW, XS>, mapW, p);
}

template <int NB, int NW>
cudaError_t launch_gemv_cfg(const CUtensorMap& mapW, const GemvParams& p, int grid,
                            cudaStream_t st) {
    // stage the activations in shared memory when they fit beside the ring
    const size_t xs_bytes = (size_t)p.M * (size_t)dec_x_row_bytes(p.G);
    if (DecCfg<NB>::kSmem + xs_bytes <= kDecSmemMax)
        return launch_gemv_nb<NB, NW, true>(mapW, p, grid, DecCfg<NB>::kSmem + xs_bytes, st);
    return launch_gemv_nb<NB, NW, false>(mapW, p, grid, DecCfg<NB>::kSmem, st);
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
    return p.M <= 8 ? launch_gemv_cfg<1, 16>(mapW, p, grid, st)
                    : launch_gemv_cfg<2, 8>(mapW, p, grid, st);
}

}  // namespace awq
