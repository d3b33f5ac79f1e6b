// W4A16 decode matmul (M <= 16 tokens) over the repacked decode tiles, and
// the repack that writes them.
//
// Decoding reads every weight once per step and is memory-bound ("AWQ:
// Activation-aware Weight Quantization ...", fdeinterviews.com/papers/awq,
// first paragraph); the OpenAlex record of the same title names weight
// packing and on-the-fly dequantisation in the inference kernels.  The plain
// packed layout (row-major words) puts the 16 rows of a slab 2-22 KB apart,
// so a kernel that streams slab by slab touches every DRAM page for a few
// hundred bytes.  The repack moves each (16-row slab, group of 128) into one
// contiguous 1088-byte tile:
//
//   bytes [0, 1024): 64 chunks of 16 bytes.  Chunk 32 h + L (h = 0, 1;
//     L = 0..31) is bytes 64 g + 16 (L % 4) .. +15 of the packed words of
//     row 16 j + L / 4 + 8 h: exactly what lane L of a warp holds as its A
//     fragments for rows L / 4 and L / 4 + 8 (decode.cuh), so a warp reads
//     a tile half with one conflict-free 16-byte load per lane.
//   bytes [1024, 1088): for r = 0..7, the fp16 scale and zero-point of row
//     16 j + r, then those of row 16 j + r + 8.
//   Tiles are ordered slab-major: tile (j, g) at byte (j G + g) 1088.  Rows
//   at or past N are zero.
//
// The tiles carry the same bytes as the plain format (a permutation of them
// when N % 16 == 0), so the kernel's algorithmic traffic is unchanged, but a
// warp's share of the matrix is now one contiguous byte range:
//
//  * Persistent grid, one CTA per SM; CTA c owns a balanced run of slabs
//    (the runs one slab longer first), i.e. a contiguous run of tiles, and
//    its warps split that run into equal contiguous ranges (intra-CTA
//    split-K where a slab is shared).
//  * Each warp streams its range through its own ring in shared memory with
//    plain 1-D bulk copies (cp.async.bulk), three tiles per stage.  No tensor
//    map is involved, so the host encodes nothing per call.
//  * With the activations staged in shared memory, the zero-point and the
//    conversion offset are folded into per-(token, group) sums formed while
//    staging (decode.cuh, folded zero-point): 4 LOP3 and 1 shift per 8
//    weights, register-sourced MMAs in one chain per group.  Otherwise (too
//    many tokens x K for shared memory) the activations come through L1 and
//    each (q - z) is formed exactly in fp16 (decode.cuh).
//  * Programmatic dependent launch and early weight fetches as in the plain
//    kernel; shared slabs are reduced through shared memory in warp order,
//    so the result is deterministic and independent of M.
#include "common.cuh"
#include "decode.cuh"
#include "kernels.cuh"

namespace awq {
namespace {

using namespace dec;

// Pipeline shape (compile-time; the defaults are the measured choice).
#ifndef AWQ_TILES_PER_STAGE
#define AWQ_TILES_PER_STAGE 3
#endif
#ifndef AWQ_TILE_STAGES_NB1
#define AWQ_TILE_STAGES_NB1 2
#endif
#ifndef AWQ_TILE_STAGES_NB2
#define AWQ_TILE_STAGES_NB2 3
#endif
#ifndef AWQ_TILE_WARPS_NB1
#define AWQ_TILE_WARPS_NB1 16
#endif
#ifndef AWQ_TILE_MINBLOCKS
#define AWQ_TILE_MINBLOCKS 1
#endif
#ifndef AWQ_TILE_EARLY_STAGES
#define AWQ_TILE_EARLY_STAGES 8
#endif
constexpr int kTilesPerStage = AWQ_TILES_PER_STAGE;
constexpr int kMaxTStages = 4;
static_assert(kTileBytes % 16 == 0 && kTile3Bytes % 16 == 0,
              "bulk copies move multiples of 16 bytes");

template <int BITS>
constexpr int tile_bytes() {
    return BITS == 4 ? kTileBytes : kTile3Bytes;
}

template <int BITS, int NB>
struct TileCfg {
    static constexpr int kTile = tile_bytes<BITS>();
    static constexpr int kStageBytes = kTilesPerStage * kTile;
    static constexpr int kWarps = NB == 1 ? AWQ_TILE_WARPS_NB1 : 8;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kStages = NB == 1 ? AWQ_TILE_STAGES_NB1 : AWQ_TILE_STAGES_NB2;
    static constexpr int kCols = 8 * NB;
    static constexpr int kSlots = 2 * kWarps;
    static constexpr size_t kRingBytes = (size_t)kWarps * kStages * kStageBytes;
    static constexpr size_t kPartBytes = (size_t)kSlots * kDecRows * kCols * sizeof(float);
    static constexpr size_t kCtlBytes =
        (size_t)kWarps * kMaxTStages * 8 + (size_t)kWarps * 12 + 16;
    static constexpr size_t kSmem = 128 + kRingBytes + kPartBytes + kCtlBytes;
};
constexpr size_t kTileSmemMax = 232448;                 // per-block opt-in limit on sm_103
static_assert(TileCfg<4, 1>::kSmem <= kTileSmemMax && TileCfg<4, 2>::kSmem <= kTileSmemMax,
              "decode kernel exceeds shared memory");

template <int NW>
struct TileCtl {
    uint64_t full[NW][kMaxTStages];
    int w_lo[NW], w_hi[NW], w_first[NW];    // each warp's tile range and first slab
    int abort;
};
static_assert(sizeof(TileCtl<TileCfg<4, 1>::kWarps>) <= TileCfg<4, 1>::kCtlBytes &&
                  sizeof(TileCtl<8>) <= TileCfg<4, 2>::kCtlBytes &&
                  TileCfg<4, 1>::kStages <= kMaxTStages && TileCfg<4, 2>::kStages <= kMaxTStages,
              "control block does not fit its shared-memory slot");

template <int BITS, int NB, int NW, bool XS>
__global__ void __launch_bounds__(NW * 32, AWQ_TILE_MINBLOCKS) gemv_tiles_kernel(const TileParams p) {
    using Cfg = TileCfg<BITS, NB>;
    static_assert(Cfg::kWarps == NW, "warp count");
    constexpr int kStages = Cfg::kStages;
    constexpr int kTStageBytes = Cfg::kStageBytes;
    constexpr int kTB = Cfg::kTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    uint8_t* ring = smem;
    float* part = reinterpret_cast<float*>(smem + Cfg::kRingBytes);
    TileCtl<NW>* ctl = reinterpret_cast<TileCtl<NW>*>(smem + Cfg::kRingBytes + Cfg::kPartBytes);
    uint8_t* xsm = smem + Cfg::kRingBytes + Cfg::kPartBytes + Cfg::kCtlBytes;   // XS only
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = p.G;

    // ---- work split: slabs over CTAs, tiles over warps ----
    // CTA-local tile indices fit in 32 bits (checked on the host).
    const int n_slabs = (int)((p.N + kDecRows - 1) / kDecRows);
    // The CTAs with one slab more come first: blocks are dispatched in index
    // order, so in a chain of programmatic launches the next kernel's heavier
    // CTAs take the SMs that this kernel's lighter CTAs free first.
    const int q = n_slabs / (int)gridDim.x, r = n_slabs - q * (int)gridDim.x;
    const int s0 = (int)blockIdx.x * q + min((int)blockIdx.x, r);
    const int s1 = s0 + q + ((int)blockIdx.x < r ? 1 : 0);
    const int U = (s1 - s0) * G;
    const int u_lo = warp_lo<NW>(U, warp), u_hi = warp_lo<NW>(U, warp + 1);
    const int n_my = u_hi - u_lo;
    const int n_st = (n_my + kTilesPerStage - 1) / kTilesPerStage;
    const int first_sl = u_lo / G;                      // this warp's first CTA-local slab
    uint8_t* my_ring = ring + (size_t)warp * kStages * kTStageBytes;
    const uint8_t* cta_tiles = p.tiles + (int64_t)s0 * G * kTB;

    // Programmatic dependent launch (see the plain decode kernel): the next
    // kernel in the stream may start at once; X and inv_s are read and Y is
    // written only after griddepcontrol.wait.  Before the wait each CTA asks
    // L2 for X and inv_s (coherent with the previous kernel's writes, which
    // are complete at the wait), and with early_weights each warp requests
    // its first ring stages -- before the CTA barrier, since the ring and
    // its mbarriers are the warp's own.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint64_t pol = l2_policy_evict_first();
    // lane 0: request stage i of this warp's range (up to kTilesPerStage
    // consecutive tiles, one contiguous copy) into ring slot s
    auto issue = [&](int i, int s) {
        const int u = u_lo + i * kTilesPerStage;
        const int nt = min(kTilesPerStage, u_hi - u);
        const uint32_t bytes = (uint32_t)(nt * kTB);
        uint64_t* bar = &ctl->full[warp][s];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(my_ring + (size_t)s * kTStageBytes, cta_tiles + (int64_t)u * kTB, bytes, bar,
                  pol);
    };
    if (warp == 0 && lane < p.M)
        bulk_prefetch_l2(p.X + (int64_t)lane * p.ldx, (uint32_t)(G * kGroup * 2));
    // (3 bits: no fused input scaling, inv_s is null)
    if (warp == 0 && lane == 31 && p.inv_s)
        bulk_prefetch_l2(p.inv_s, (uint32_t)(G * kGroup * 4));
    const int n_first = min(kStages, n_st);
    const int n_early = p.early_weights ? min(n_first, AWQ_TILE_EARLY_STAGES) : 0;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&ctl->full[warp][s], 1);
        fence_mbar_init();
        ctl->w_lo[warp] = u_lo;
        ctl->w_hi[warp] = u_hi;
        ctl->w_first[warp] = first_sl;
        for (int i = 0; i < n_early; ++i) issue(i, i);
    }
    if (threadIdx.x == 0) ctl->abort = 0;
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (lane == 0)
        for (int i = n_early; i < n_first; ++i) issue(i, i);
    __syncwarp();

    const uint8_t* xs[NB];
    uint8_t* bs = nullptr;
    if constexpr (XS) {
        const int64_t xrow = BITS == 4 ? dec_x_row_bytes(G) : dec_x3_row_bytes((int64_t)G * kGroup);
        if constexpr (BITS == 4) {
            bs = xsm + (int64_t)p.M * xrow;
            stage_x_folded<NB>(xsm, bs, p.X, p.ldx, p.M, p.inv_s, G, threadIdx.x, Cfg::kThreads);
        } else {
            stage_x3(xsm, p.X, p.ldx, p.M, (int64_t)G * kGroup, threadIdx.x, Cfg::kThreads);
        }
        __syncthreads();
        // lanes of absent tokens read the last token's row; their outputs
        // are dropped
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) xs[nb] = xsm + min(g + 8 * nb, p.M - 1) * xrow;
    } else {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) xs[nb] = nullptr;
    }

    // a finished slab goes straight to Y when this warp owns all its tiles,
    // else into this warp's first/last partial slot
    auto flush = [&](int sl, const float (&y)[NB][4]) {
        const bool owned = sl * G >= u_lo && (sl + 1) * G <= u_hi;
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
    int sl = first_sl, gi = u_lo - first_sl * G;        // (slab, group) of the next tile
    int i = 0;
    bool ok = true;
    for (; i < n_st; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&ctl->full[warp][s], (uint32_t)(i / kStages) & 1u, &ctl->abort,
                       p.status)) {
            ok = false;
            break;
        }
        const uint8_t* stage = my_ring + (size_t)s * kTStageBytes;
        const int nt = min(kTilesPerStage, u_hi - (u_lo + i * kTilesPerStage));
#pragma unroll
        for (int jt = 0; jt < kTilesPerStage; ++jt) {
            if (jt < nt) {
                if (sl != cur) {
                    if (cur >= 0) flush(cur, y);
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int j = 0; j < 4; ++j) y[nb][j] = 0.0f;
                    cur = sl;
                }
                const uint8_t* tile = stage + jt * kTB;
                if constexpr (BITS == 4) {
                    const uint4 wa = *reinterpret_cast<const uint4*>(tile + lane * 16);
                    const uint4 wb = *reinterpret_cast<const uint4*>(tile + 512 + lane * 16);
                    const uint2 sz = *reinterpret_cast<const uint2*>(tile + 1024 + g * 8);
                    if constexpr (XS) {
                        group_mma_folded<NB>(y, sz, wa, wb, xs, bs, gi, t);
                    } else {
                        GroupX<NB> gx;
                        load_group_x<NB>(gx, p.X, p.ldx, p.M, p.inv_s, gi, g, t);
                        group_mma<NB, false>(y, (uint16_t)(sz.x & 0xFFFFu),
                                             (uint16_t)(sz.y & 0xFFFFu), (uint16_t)(sz.x >> 16),
                                             (uint16_t)(sz.y >> 16), gx, wa, wb, xs, gi, t);
                    }
                } else {
                    // rows g and g + 8: 48 bytes of planes each, then the scales
                    const uint4* ra = reinterpret_cast<const uint4*>(tile + 48 * g);
                    const uint4* rb = reinterpret_cast<const uint4*>(tile + 48 * (g + 8));
                    const uint4 a0 = ra[0], a1 = ra[1], a2 = ra[2];
                    const uint4 b0 = rb[0], b1 = rb[1], b2 = rb[2];
                    const uint32_t A[12] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y,
                                            a1.z, a1.w, a2.x, a2.y, a2.z, a2.w};
                    const uint32_t B[12] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y,
                                            b1.z, b1.w, b2.x, b2.y, b2.z, b2.w};
                    const uint2 sz = *reinterpret_cast<const uint2*>(tile + 768 + g * 8);
                    group_mma3<NB, XS>(y, sz, A, B, xs, p.X, p.ldx, p.M, gi, g, t);
                }
                if (++gi == G) {
                    gi = 0;
                    ++sl;
                }
            }
        }
        __syncwarp();
        if (lane == 0 && i + kStages < n_st) {
            // the warp's reads of this stage are done; the copy may overwrite it
            fence_proxy_async_smem();
            issue(i + kStages, s);
        }
    }
    if (ok && cur >= 0) flush(cur, y);
    if (!ok && lane == 0) {
        // bounded drain of the copies this warp still has in flight
        for (int k = i; k < n_st && k < i + kStages; ++k) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&ctl->full[warp][k % kStages], (uint32_t)(k / kStages) & 1u))
                if (globaltimer_ns() - t0 > 100000000ull) break;
        }
    }
    __syncthreads();
    if (ctl->abort) return;

    // ---- slabs shared by several warps: add the partials in warp order ----
    if (warp >= 1 && u_lo < U && u_lo % G != 0) {
        const int rsl = u_lo / G;
        if (ctl->w_lo[warp - 1] <= rsl * G) {
            const int64_t row0 = (int64_t)(s0 + rsl) * kDecRows;
            for (int e = lane; e < kDecRows * p.M; e += 32) {
                const int r = e / p.M, m = e - r * p.M;
                float acc = 0.0f;
                for (int j = 0; j < NW; ++j) {
                    const int lo = ctl->w_lo[j], hi = ctl->w_hi[j];
                    if (hi <= lo || hi <= rsl * G || lo >= (rsl + 1) * G) continue;
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

template <int BITS, int NB, int NW, bool XS>
cudaError_t launch_tiles_nb(const TileParams& p, int grid, size_t smem, cudaStream_t st) {
    cudaError_t e = smem_attr_once<gemv_tiles_kernel<BITS, NB, NW, XS>>((int)kTileSmemMax);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(TileCfg<BITS, NB>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_tiles_kernel<BITS, NB, NW, XS>, p);
}

template <int BITS, int NB, int NW>
cudaError_t launch_tiles_cfg(const TileParams& p, int grid, cudaStream_t st) {
    using Cfg = TileCfg<BITS, NB>;
    const size_t xs_bytes =
        BITS == 4 ? (size_t)p.M * (size_t)dec_x_row_bytes(p.G) + (size_t)dec_bs_bytes(p.G, NB)
                  : (size_t)p.M * (size_t)dec_x3_row_bytes((int64_t)p.G * kGroup);
    if (Cfg::kSmem + xs_bytes <= kTileSmemMax)
        return launch_tiles_nb<BITS, NB, NW, true>(p, grid, Cfg::kSmem + xs_bytes, st);
    return launch_tiles_nb<BITS, NB, NW, false>(p, grid, Cfg::kSmem, st);
}

// One thread per 16 bytes of the tiled buffer (68 per tile): consecutive
// threads write consecutive bytes.  I is the chunk index type: 32-bit
// whenever the chunk count fits (its divisions are several times cheaper),
// else 64-bit.
template <typename I>
__global__ void __launch_bounds__(256)
    repack_int4_kernel(const uint32_t* __restrict__ qweight, const uint16_t* __restrict__ scales,
                       const uint16_t* __restrict__ zeros, int64_t N, int64_t K,
                       uint4* __restrict__ tiles, int64_t n_chunks) {
    constexpr int kChunks = kTileBytes / 16;            // 68
    const I G = (I)(K / kGroup);
    for (I u = (I)blockIdx.x * blockDim.x + threadIdx.x; u < (I)n_chunks;
         u += (I)gridDim.x * blockDim.x) {
        const I tile = u / kChunks;
        const int c = (int)(u - tile * kChunks);
        const int64_t j = tile / G, gi = tile - (I)j * G;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (c < 64) {
            const int h = c >> 5, L = c & 31;
            const int64_t row = j * kDecRows + (L >> 2) + 8 * h;
            if (row < N)
                v = __ldg(reinterpret_cast<const uint4*>(qweight + row * (K / 8) + gi * 16 +
                                                         (L & 3) * 4));
        } else {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int64_t ra = j * kDecRows + (c - 64) * 2 + e, rb = ra + 8;
                const uint32_t sa = ra < N ? scales[ra * G + gi] : 0u;
                const uint32_t za = ra < N ? zeros[ra * G + gi] : 0u;
                const uint32_t sb = rb < N ? scales[rb * G + gi] : 0u;
                const uint32_t zb = rb < N ? zeros[rb * G + gi] : 0u;
                w[2 * e] = sa | (za << 16);
                w[2 * e + 1] = sb | (zb << 16);
            }
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        tiles[u] = v;
    }
}

// The 3-bit tiles: one thread per 16 bytes (52 per tile): 48 chunks of the
// 16 rows' planes (row r's 48 bytes at 48 r), then the four of scales and
// zero-points.
template <typename I>
__global__ void __launch_bounds__(256)
    repack_int3_kernel(const uint32_t* __restrict__ planes, const uint16_t* __restrict__ scales,
                       const uint16_t* __restrict__ zeros, int64_t N, int64_t K,
                       uint4* __restrict__ tiles, int64_t n_chunks) {
    constexpr int kChunks = kTile3Bytes / 16;           // 52
    const I G = (I)(K / kGroup);
    const int64_t wrow = K / 32 * 3;
    for (I u = (I)blockIdx.x * blockDim.x + threadIdx.x; u < (I)n_chunks;
         u += (I)gridDim.x * blockDim.x) {
        const I tile = u / kChunks;
        const int c = (int)(u - tile * kChunks);
        const int64_t j = tile / G, gi = tile - (I)j * G;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (c < 48) {
            const int64_t row = j * kDecRows + c / 3;
            if (row < N)
                v = __ldg(reinterpret_cast<const uint4*>(planes + row * wrow + gi * 12 + (c % 3) * 4));
        } else {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int64_t ra = j * kDecRows + (c - 48) * 2 + e, rb = ra + 8;
                const uint32_t sa = ra < N ? scales[ra * G + gi] : 0u;
                const uint32_t za = ra < N ? zeros[ra * G + gi] : 0u;
                const uint32_t sb = rb < N ? scales[rb * G + gi] : 0u;
                const uint32_t zb = rb < N ? zeros[rb * G + gi] : 0u;
                w[2 * e] = sa | (za << 16);
                w[2 * e + 1] = sb | (zb << 16);
            }
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        tiles[u] = v;
    }
}

}  // namespace

cudaError_t launch_repack_int3(const uint32_t* planes, const uint16_t* scales,
                               const uint16_t* zeros, int64_t N, int64_t K, void* tiles,
                               int num_sms, cudaStream_t st) {
    const int64_t n_chunks = (N + kDecRows - 1) / kDecRows * (K / kGroup) * (kTile3Bytes / 16);
    if (n_chunks == 0) return cudaSuccess;
    int64_t blocks = (n_chunks + 255) / 256;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    if (n_chunks + (int64_t)blocks * 256 < (1LL << 32))
        repack_int3_kernel<uint32_t><<<(unsigned)blocks, 256, 0, st>>>(
            planes, scales, zeros, N, K, static_cast<uint4*>(tiles), n_chunks);
    else
        repack_int3_kernel<int64_t><<<(unsigned)blocks, 256, 0, st>>>(
            planes, scales, zeros, N, K, static_cast<uint4*>(tiles), n_chunks);
    return cudaGetLastError();
}

cudaError_t launch_gemv_tiles(const TileParams& p, int num_sms, cudaStream_t st) {
    if (p.M <= 0 || p.N <= 0) return cudaSuccess;
    const int64_t n_slabs = (p.N + kDecRows - 1) / kDecRows;
    const int grid = (int)(n_slabs < num_sms ? n_slabs : num_sms);
    // the kernel indexes a CTA's tiles in 32 bits
    if ((n_slabs / grid + 1) * (int64_t)p.G >= (1LL << 31)) return cudaErrorInvalidValue;
    if (p.bits == 3)
        return p.M <= 8 ? launch_tiles_cfg<3, 1, TileCfg<3, 1>::kWarps>(p, grid, st)
                        : launch_tiles_cfg<3, 2, 8>(p, grid, st);
    return p.M <= 8 ? launch_tiles_cfg<4, 1, TileCfg<4, 1>::kWarps>(p, grid, st)
                    : launch_tiles_cfg<4, 2, 8>(p, grid, st);
}

cudaError_t launch_repack_int4(const uint32_t* qweight, const uint16_t* scales,
                               const uint16_t* zeros, int64_t N, int64_t K, void* tiles,
                               int num_sms, cudaStream_t st) {
    const int64_t n_chunks = (N + kDecRows - 1) / kDecRows * (K / kGroup) * (kTileBytes / 16);
    if (n_chunks == 0) return cudaSuccess;
    int64_t blocks = (n_chunks + 255) / 256;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    if (n_chunks + (int64_t)blocks * 256 < (1LL << 32))
        repack_int4_kernel<uint32_t><<<(unsigned)blocks, 256, 0, st>>>(
            qweight, scales, zeros, N, K, static_cast<uint4*>(tiles), n_chunks);
    else
        repack_int4_kernel<int64_t><<<(unsigned)blocks, 256, 0, st>>>(
            qweight, scales, zeros, N, K, static_cast<uint4*>(tiles), n_chunks);
    return cudaGetLastError();
}

}  // namespace awq
