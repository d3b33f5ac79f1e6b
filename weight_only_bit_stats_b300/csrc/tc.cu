// Tensor-core kernels on sm_103a (tcgen05 MMA, TMEM accumulators, TMA):
//
//  * W4A16 GEMM for M > 16 tokens: Y = X deq(Wq)^T.  Under large batches the
//    matmul becomes compute-bound ("AWQ: Activation-aware Weight Quantization
//    ...", fdeinterviews.com/papers/awq, ninth paragraph); the packed tile is
//    dequantised on the fly into shared memory and multiplied on the tensor
//    cores (the OpenAlex record's abstract: on-the-fly dequantisation, kernel
//    fusion).
//  * The alpha search (third paragraph: grid search over alpha on a small
//    calibration set): per alpha, the producer fake-quantises W diag(s) with
//    the exact rounding of the packer and writes the residual
//    E = Q(W diag(s)) diag(s)^-1 - W as fp16; the tensor cores form Xcal E^T
//    and the epilogue reduces its squares -- the per-alpha output MSE is a
//    fused epilogue and E never reaches global memory.
//  * The same search through the Gram matrix: ||Xcal E^T||^2 = tr(E G E^T)
//    with G = Xcal^T Xcal, so with G/T (fp16, [K, K]) in place of the
//    calibration tokens the tensor cores form E (G/T), and the epilogue
//    multiplies each accumulator column by the matching residual column --
//    recomputed from W, s and the group parameters the producer exports --
//    and adds.  The pages' grid search leaves the evaluation route open; this
//    one costs 2 N K^2 per alpha instead of 2 T N K.
//  * G/T itself: a plain fp16 GEMM of X^T with itself (both operands by TMA
//    from a transposed copy of Xcal), scaled by 1/T and rounded to fp16.
//
// One persistent CTA per SM.  Warp roles:
//   warp 0      TMA producer of activation tiles (one thread)
//   warp 1      MMA issuer (one thread): tcgen05.mma M=128 N=256 K=16
//   warp 2      TMEM allocator (512 columns = two 256-column accumulators)
//   warps 4..7  epilogue: tcgen05.ld of their TMEM lane quarter
//   warps 8..   weight-operand producers (dequant or fake-quant)
// Work item = 128 weight rows x (256 tokens for the GEMM, 512 for the
// search, i.e. both accumulators), looping over K in groups of 128.
// Operand tiles are K-major in the 128-byte swizzled layout; the A tile of
// a group is two [128 x 64] sub-tiles, the B tile two [256 x 64] sub-tiles.
// Every mbarrier wait is bounded; a timeout sets an abort flag that every
// role checks, records AWQ's timeout status, and the CTA exits cleanly after
// its own TMA copies and MMAs have drained and TMEM is freed.
#include "common.cuh"
#include "kernels.cuh"

namespace awq {
namespace {

enum { kModeGemm = 0, kModeSearch = 1, kModeXtX = 2, kModeGram = 3, kModeGemm3 = 4 };

constexpr int kNA = 2;                            // A (weight) stages
constexpr int kNB = 2;                            // B (activation) stages
constexpr int kNW = 3;                            // GEMM packed-word stages
constexpr int kWStage = kTcRows * 64;             // 8 KB: one group of 128 packed rows
constexpr int kAStage = kTcRows * kGroup * 2;     // 32 KB
constexpr int kASub = kTcRows * 64 * 2;           // 16 KB
constexpr int kBStage = kTcTokens * kGroup * 2;   // 64 KB
constexpr int kBSub = kTcTokens * 64 * 2;         // 32 KB
constexpr int kTmemCols = 512;

constexpr int kWarpTma = 0, kWarpMma = 1, kWarpTmem = 2, kWarpTmaW = 3, kWarpEpi0 = 4,
              kWarpProd0 = 8;

// The two W4A16 / W3A16 GEMM modes share everything but the producer.
template <int MODE>
constexpr bool is_gemm() {
    return MODE == kModeGemm || MODE == kModeGemm3;
}

template <int MODE>
struct Cfg {
    static constexpr int kProdWarps = is_gemm<MODE>() ? 4 : (MODE == kModeXtX ? 0 : 16);
    static constexpr int kThreads = (kWarpProd0 + kProdWarps) * 32;
    static constexpr int kHalves = is_gemm<MODE>() ? 1 : 2;     // accumulators per item
};

struct SmemCtl {
    uint64_t w_full[kNW], w_empty[kNW];     // GEMM: packed-word ring
    uint64_t a_full[kNA], a_empty[kNA];
    uint64_t b_full[kNB], b_empty[kNB];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t par_full[2], par_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

// Shared memory per mode (the rest of the SM's 228 KB stays L1, which the
// GEMM producer's packed-word loads and the search producer's scale loads
// go through).
template <int MODE>
constexpr size_t ring_w_bytes() {
    return MODE == kModeGemm ? (size_t)kNW * kWStage : 0;
}
template <int MODE>
constexpr size_t smem_bytes() {
    return 1024 /*align slack*/ + (size_t)kNA * kAStage + (size_t)kNB * kBStage +
           ring_w_bytes<MODE>() + sizeof(SmemCtl);
}

struct Item {
    int n_tile, t_tile, alpha;
    int split, g0, g1;                 // GEMM split-K: this item's groups [g0, g1)
    int slot;                          // GEMM stream-K share: partial slot, else -1
};

template <int MODE>
__device__ __forceinline__ Item decode_item(int item, const TcParams& p) {
    Item it;
    if (is_gemm<MODE>()) {
        // token tiles in bands of up to 8 (2048 tokens): within a band,
        // consecutive CTAs share a weight tile (the band's token tiles of one
        // weight tile run together) and the weight tiles go round, so the
        // band's activations stay in L2 while the packed words stream by,
        // once per band
        const int per_split = p.t_tiles * p.n_tiles;
        it.split = item / per_split;
        const int q = item - it.split * per_split;
        const int band_tiles = p.t_tiles < 8 ? p.t_tiles : 8;
        const int band = q / (band_tiles * p.n_tiles);
        const int rb = q - band * band_tiles * p.n_tiles;
        const int bt = (band + 1) * band_tiles <= p.t_tiles ? band_tiles
                                                            : p.t_tiles - band * band_tiles;
        it.t_tile = band * band_tiles + rb % bt;
        it.n_tile = rb / bt;
        it.alpha = 0;
        it.g0 = (int)((int64_t)it.split * p.G / p.k_splits);
        it.g1 = (int)((int64_t)(it.split + 1) * p.G / p.k_splits);
    } else if (MODE == kModeXtX) {     // (row tile, column block) of X^T X
        it.alpha = 0;
        it.t_tile = item % p.t_tiles;
        it.n_tile = item / p.t_tiles;
        it.split = 0;
        it.g0 = 0;
        it.g1 = p.G;
    } else {                           // consecutive CTAs share the weight tile
        it.alpha = item % p.n_alpha;
        const int rest = item / p.n_alpha;
        it.t_tile = rest % p.t_tiles;
        it.n_tile = rest / p.t_tiles;
        it.split = 0;
        it.g0 = 0;
        it.g1 = p.G;
    }
    return it;
}

// Stream-K tail share of CTA c (0 <= c < sk_ctas): units [s0, s1) of the
// tail's sk_tiles * G (tile, group) units, tile-major, s_c = c * units /
// sk_ctas.  A share is shorter than one tile's G groups, so it covers the
// end of one tile and possibly the start of the next.
__host__ __device__ __forceinline__ void sk_share(int c, int sk_ctas, int sk_tiles, int G,
                                                  int64_t& s0, int64_t& s1) {
    const int64_t units = (int64_t)sk_tiles * G;
    s0 = (int64_t)c * units / sk_ctas;
    s1 = (int64_t)(c + 1) * units / sk_ctas;
}

// This CTA's i-th item; false past its last.  Items go round the CTAs
// (item blockIdx.x + i gridDim.x), except under a GEMM stream-K tail, where
// the CTA takes whole tiles blockIdx.x + i sk_ctas of the first sk_full,
// then its tail share (one or two pieces, partial slots 2 c and 2 c + 1).
template <int MODE>
__device__ __forceinline__ bool cta_item(int i, const TcParams& p, Item& it) {
    if (is_gemm<MODE>() && p.sk_tiles > 0) {
        const int c = blockIdx.x, nf = p.sk_full / p.sk_ctas;
        if (i < nf) {
            it = decode_item<MODE>(c + i * p.sk_ctas, p);
            it.slot = -1;
            return true;
        }
        int64_t s0, s1;
        sk_share(c, p.sk_ctas, p.sk_tiles, p.G, s0, s1);
        if (s0 >= s1) return false;
        const int ta = (int)(s0 / p.G);
        const int64_t a_end = min(s1, (int64_t)(ta + 1) * p.G);
        int tile, g0, g1;
        if (i == nf) {
            tile = ta;
            g0 = (int)(s0 - (int64_t)ta * p.G);
            g1 = (int)(a_end - (int64_t)ta * p.G);
        } else if (i == nf + 1 && s1 > a_end) {
            tile = ta + 1;
            g0 = 0;
            g1 = (int)(s1 - (int64_t)(ta + 1) * p.G);
        } else {
            return false;
        }
        it = decode_item<MODE>(p.sk_full + tile, p);
        it.g0 = g0;
        it.g1 = g1;
        it.slot = 2 * c + (i - nf);
        return true;
    }
    const int item = blockIdx.x + i * gridDim.x;
    if (item >= p.n_items) return false;
    it = decode_item<MODE>(item, p);
    it.slot = -1;
    return true;
}

__device__ __forceinline__ uint32_t pack_h2_rn(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Bounded wait that ignores the abort flag (used only to drain own copies).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 100000000ull) break;
    }
}

// ---- role: TMA producer of activation tiles ----
template <int MODE>
__device__ void role_tma(const CUtensorMap* mapX, const CUtensorMap* mapA, const TcParams& p,
                         uint8_t* As, uint8_t* Bs, SmemCtl* ctl) {
    constexpr int H = Cfg<MODE>::kHalves;
    volatile int* abort = &ctl->abort;
    // the activation tiles are re-read by every weight tile: keep them in L2
    const uint64_t pol = l2_policy_evict_last();
    uint32_t a_iter = 0, b_iter = 0;
    Item it;
    for (int li = 0; cta_item<MODE>(li, p, it); ++li) {
        const int t0 = it.t_tile * kTcTokens * H;
        for (int g = it.g0; g < it.g1; ++g) {
            if constexpr (MODE == kModeXtX) {
                // the A operand is a tile of the same transposed matrix
                const int st = a_iter % kNA;
                if (!mbar_wait(&ctl->a_empty[st], ((a_iter / kNA) & 1u) ^ 1u, abort, p.status))
                    goto drain;
                mbar_arrive_expect_tx(&ctl->a_full[st], kAStage);
                uint8_t* dst = As + st * kAStage;
                tma_load_2d_hint(dst, mapA, &ctl->a_full[st], g * kGroup, it.n_tile * kTcRows, pol);
                tma_load_2d_hint(dst + kASub, mapA, &ctl->a_full[st], g * kGroup + 64,
                                 it.n_tile * kTcRows, pol);
                ++a_iter;
            }
            for (int h = 0; h < H; ++h) {
                const int st = b_iter % kNB;
                const uint32_t ph = (b_iter / kNB) & 1u;
                if (!mbar_wait(&ctl->b_empty[st], ph ^ 1u, abort, p.status)) goto drain;
                mbar_arrive_expect_tx(&ctl->b_full[st], kBStage);
                uint8_t* dst = Bs + st * kBStage;
                tma_load_2d_hint(dst, mapX, &ctl->b_full[st], g * kGroup, t0 + h * kTcTokens, pol);
                tma_load_2d_hint(dst + kBSub, mapX, &ctl->b_full[st], g * kGroup + 64,
                                 t0 + h * kTcTokens, pol);
                ++b_iter;
            }
        }
    }
    return;
drain:
    // wait (bounded) for the copies this thread issued into each stage
    for (int d = 1; d <= kNB && (int)b_iter - d >= 0; ++d) {
        const uint32_t i = b_iter - d;
        mbar_drain(&ctl->b_full[i % kNB], (i / kNB) & 1u);
    }
    if constexpr (MODE == kModeXtX) {
        for (int d = 1; d <= kNA && (int)a_iter - d >= 0; ++d) {
            const uint32_t i = a_iter - d;
            mbar_drain(&ctl->a_full[i % kNA], (i / kNA) & 1u);
        }
    }
}

// ---- role: packed-weight TMA (GEMM) ----
// One box per (item, group): the group's 16 packed words of the tile's 128
// rows (rows past N read as zero), 64-byte swizzle, into the kNW-stage ring
// the producer warps dequantise from.
__device__ void role_tma_w(const CUtensorMap* mapW, const TcParams& p, uint8_t* Ws,
                           SmemCtl* ctl) {
    volatile int* abort = &ctl->abort;
    uint32_t w_iter = 0;
    Item it;
    for (int li = 0; cta_item<kModeGemm>(li, p, it); ++li) {
        for (int g = it.g0; g < it.g1; ++g) {
            const int st = w_iter % kNW;
            if (!mbar_wait(&ctl->w_empty[st], ((w_iter / kNW) & 1u) ^ 1u, abort, p.status))
                goto drain;
            mbar_arrive_expect_tx(&ctl->w_full[st], kWStage);
            tma_load_2d(Ws + st * kWStage, mapW, &ctl->w_full[st], g * (kGroup / 8),
                        it.n_tile * kTcRows);
            ++w_iter;
        }
    }
    return;
drain:
    // wait (bounded) for the copies this thread issued into each stage
    for (int d = 1; d <= kNW && (int)w_iter - d >= 0; ++d) {
        const uint32_t i = w_iter - d;
        mbar_drain(&ctl->w_full[i % kNW], (i / kNW) & 1u);
    }
}

// ---- role: MMA issuer ----
template <int MODE>
__device__ void role_mma(const TcParams& p, uint8_t* As, uint8_t* Bs, SmemCtl* ctl, uint32_t tmem) {
    constexpr int H = Cfg<MODE>::kHalves;
    constexpr uint32_t idesc = umma_idesc_f16_f32(kTcRows, kTcTokens);
    volatile int* abort = &ctl->abort;
    uint32_t a_iter = 0, b_iter = 0, acc_iter = 0;
    Item it;
    for (int li = 0; cta_item<MODE>(li, p, it); ++li) {
        for (int g = it.g0; g < it.g1; ++g) {
            const int sa = a_iter % kNA;
            if (!mbar_wait(&ctl->a_full[sa], (a_iter / kNA) & 1u, abort, p.status)) goto out;
            tc_fence_after();
            const uint32_t a_base = smem_u32(As + sa * kAStage);
            for (int h = 0; h < H; ++h) {
                const uint32_t slot_iter = acc_iter + h;
                const int slot = slot_iter & 1;
                if (g == it.g0) {
                    if (!mbar_wait(&ctl->acc_empty[slot], ((slot_iter >> 1) & 1u) ^ 1u, abort,
                                   p.status))
                        goto out;
                    tc_fence_after();
                }
                const int sb = b_iter % kNB;
                if (!mbar_wait(&ctl->b_full[sb], (b_iter / kNB) & 1u, abort, p.status)) goto out;
                tc_fence_after();
                const uint32_t b_base = smem_u32(Bs + sb * kBStage);
                const uint32_t d = tmem + (uint32_t)(slot * kTcTokens);
#pragma unroll
                for (int ks = 0; ks < kGroup / 16; ++ks) {
                    const uint32_t sub = ks >> 2, koff = (ks & 3) * 32;
                    const uint64_t ad = umma_desc_sw128(a_base + sub * kASub + koff);
                    const uint64_t bd = umma_desc_sw128(b_base + sub * kBSub + koff);
                    umma_f16(d, ad, bd, idesc, (g > it.g0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(&ctl->b_empty[sb]);
                ++b_iter;
            }
            umma_commit(&ctl->a_empty[sa]);
            ++a_iter;
        }
        for (int h = 0; h < H; ++h) umma_commit(&ctl->acc_full[(acc_iter + h) & 1]);
        acc_iter += H;
    }
out:
    // every MMA this thread issued has finished before TMEM is released
    umma_commit(&ctl->mma_done);
    mbar_drain(&ctl->mma_done, 0);
}

// ---- role: epilogue ----
template <int MODE>
__device__ void role_epilogue(const TcParams& p, SmemCtl* ctl, uint32_t tmem, int q, int lane) {
    constexpr int H = Cfg<MODE>::kHalves;
    volatile int* abort = &ctl->abort;
    uint32_t acc_iter = 0, item_iter = 0;
    Item it;
    for (int li = 0; cta_item<MODE>(li, p, it); ++li, ++item_iter) {
        const int64_t n = (int64_t)it.n_tile * kTcRows + q * 32 + lane;   // this thread's row
        const int r = q * 32 + lane;                                       // row within the tile
        float sq = 0.0f;
        double dsum = 0.0;
        for (int h = 0; h < H; ++h) {
            const int slot = acc_iter & 1;
            if (!mbar_wait(&ctl->acc_full[slot], (acc_iter >> 1) & 1u, abort, p.status)) return;
            tc_fence_after();
            if (MODE == kModeGram && h == 0) {
                if (!mbar_wait(&ctl->par_full[item_iter & 1], (item_iter >> 1) & 1u, abort,
                               p.status))
                    return;
            }
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * kTcTokens);
            const int64_t tok0 = ((int64_t)it.t_tile * H + h) * kTcTokens;
#pragma unroll 1
            for (int c = 0; c < kTcTokens / 32; ++c) {
                if constexpr (MODE == kModeGram) {
                    // sum over these 32 columns of (E (G/T))[n, col] E[n, col],
                    // E being the fp16 residuals the producer exported for
                    // this item's columns (the values the tensor cores
                    // multiplied), 8 columns at a time
                    const int64_t col = tok0 + c * 32;
                    if (col < p.K) {                           // uniform over the warp
                        const uint4* er = reinterpret_cast<const uint4*>(
                            p.e_exp +
                            ((int64_t)(blockIdx.x * 2 + (item_iter & 1)) * kTcRows + r) *
                                kSearchTokensPerItem +
                            (col - (int64_t)it.t_tile * kSearchTokensPerItem));
                        uint4 e4[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) e4[j] = __ldcg(er + j);
                        float v[32];
                        tmem_ld32(taddr + c * 32, v);
                        float acc = 0.0f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const __half2* hh = reinterpret_cast<const __half2*>(&e4[j]);
                            float a8 = 0.0f;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __half22float2(hh[e]);
                                a8 = fmaf(v[8 * j + 2 * e], f.x, a8);
                                a8 = fmaf(v[8 * j + 2 * e + 1], f.y, a8);
                            }
                            acc += a8;
                        }
                        if (n < p.N) dsum += (double)acc;
                    }
                    continue;
                }
                float v[32];
                tmem_ld32(taddr + c * 32, v);
                if (is_gemm<MODE>()) {
                    if (n < p.N) {
                        if (it.slot >= 0) {
                            // stream-K share: fp32 partial tile [token][row]
                            float* wsp = p.ws_sk + (int64_t)it.slot * (kTcRows * kTcTokens) +
                                         (int64_t)(c * 32) * kTcRows + r;
#pragma unroll
                            for (int j = 0; j < 32; ++j) wsp[j * kTcRows] = v[j];
                        } else if (p.k_splits == 1) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int64_t tok = tok0 + c * 32 + j;
                                if (tok < p.rows_tok)      // streaming: Y does not evict X
                                    __stcs(reinterpret_cast<unsigned short*>(p.Y) + tok * p.ldy + n,
                                           __half_as_ushort(__float2half_rn(v[j])));
                            }
                        } else {
                            // fp32 partial of this split, laid out like Y
                            float* wsp = p.ws_partial + (int64_t)it.split * p.rows_tok * p.N + n;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int64_t tok = tok0 + c * 32 + j;
                                if (tok < p.rows_tok) __stcs(wsp + tok * p.N, v[j]);
                            }
                        }
                    }
                } else if (MODE == kModeXtX) {
                    // G/T: 32 consecutive columns of row n, as fp16
                    const int64_t col = tok0 + c * 32;
                    if (n < p.N && col < p.rows_tok) {
                        uint32_t w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            w[j] = pack_h2_rn(v[2 * j] * p.inv_t, v[2 * j + 1] * p.inv_t);
                        uint4* dst = reinterpret_cast<uint4*>(p.gout + n * p.rows_tok + col);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) sq = fmaf(v[j], v[j], sq);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->acc_empty[slot]);
            ++acc_iter;
        }
        if (MODE == kModeGram) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->par_empty[item_iter & 1]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
            if (lane == 0)
                p.partials[(((int64_t)it.alpha * p.n_tiles + it.n_tile) * p.t_tiles + it.t_tile) * 4 +
                           q] = dsum;
        }
        if (MODE == kModeSearch) {
            // one fp64 partial per epilogue warp; the final reduction adds
            // them in a fixed order
            double d = (double)sq;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0)
                p.partials[(((int64_t)it.alpha * p.n_tiles + it.n_tile) * p.t_tiles + it.t_tile) * 4 +
                           q] = d;
        }
    }
}

// ---- role: GEMM weight producer (int4 -> fp16 (q - z) * scale) ----
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
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// 8 nibbles -> 8 consecutive fp16 values of (q - z) * scale.  (q - z), an
// integer in [-15, 15], is exact in fp16; its product with the fp16 scale can
// need up to 15 significant bits and is rounded once to fp16 (relative error
// at most 2^-11, the rounding an fp16 weight carries anyway).
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 z1024, __half2 zneg64, __half2 sc) {
    const uint32_t magic = 0x64006400u;
    const __half2 sixteenth = __half2half2(__float2half_rn(0.0625f));
    const uint32_t w8 = w >> 8;
    __half2 p0 = __hsub2(u2h(lop3_and_or(w, 0x000F000Fu, magic)), z1024);           // e0 | e4
    __half2 p1 = __hfma2(u2h(lop3_and_or(w, 0x00F000F0u, magic)), sixteenth, zneg64);  // e1 | e5
    __half2 p2 = __hsub2(u2h(lop3_and_or(w8, 0x000F000Fu, magic)), z1024);          // e2 | e6
    __half2 p3 = __hfma2(u2h(lop3_and_or(w8, 0x00F000F0u, magic)), sixteenth, zneg64); // e3 | e7
    const uint32_t u0 = h2u(__hmul2(p0, sc)), u1 = h2u(__hmul2(p1, sc));
    const uint32_t u2 = h2u(__hmul2(p2, sc)), u3 = h2u(__hmul2(p3, sc));
    return make_uint4(prmt(u0, u1, 0x5410), prmt(u2, u3, 0x5410), prmt(u0, u1, 0x7632),
                      prmt(u2, u3, 0x7632));
}

// Hint: bring the 128-byte line holding ptr into L2.
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// 3-bit GEMM producer: groups of plane words a row requests into L2 ahead of
// its own loads (which run one group ahead): with ~0.7 us of MMA work per
// group, six groups cover a DRAM miss several times over.  (The 4-bit
// producer reads its words from the TMA ring instead.)
constexpr int kProdPrefetch = 6;

__device__ void role_prod_gemm(const TcParams& p, uint8_t* As, const uint8_t* Ws, SmemCtl* ctl,
                               int r, int lane) {
    volatile int* abort = &ctl->abort;
    // this row's 16-byte chunk j of a ring stage (64-byte swizzle)
    const uint32_t wrow = (uint32_t)r * 64u, wx = (uint32_t)((r >> 1) & 3);
    uint32_t a_iter = 0, w_iter = 0;
    Item it;
    for (int li = 0; cta_item<kModeGemm>(li, p, it); ++li) {
        const int64_t n = (int64_t)it.n_tile * kTcRows + r;
        const bool valid = n < p.N;
        const uint16_t* srow = p.scales + (valid ? n : 0) * p.G;
        const uint16_t* zrow = p.zeros + (valid ? n : 0) * p.G;
        uint16_t csc = 0, cze = 0;
        if (valid) {
            csc = __ldg(srow + it.g0);
            cze = __ldg(zrow + it.g0);
            // the row's scales and zero-points of this item
            for (int g = it.g0; g < it.g1; g += 64) {
                prefetch_l2(srow + g);
                prefetch_l2(zrow + g);
            }
        }
        for (int g = it.g0; g < it.g1; ++g) {
            uint16_t nsc = 0, nze = 0;
            if (valid && g + 1 < it.g1) {
                nsc = __ldg(srow + g + 1);
                nze = __ldg(zrow + g + 1);
            }
            // the group's packed words of this row, from the TMA ring
            const int sw = w_iter % kNW;
            if (!mbar_wait(&ctl->w_full[sw], (w_iter / kNW) & 1u, abort, p.status)) return;
            const uint8_t* wst = Ws + sw * kWStage + wrow;
            uint4 cur[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                cur[j] = *reinterpret_cast<const uint4*>(wst + (((uint32_t)j ^ wx) << 4));
            // the stage's next fill is an async-proxy write: order these
            // generic-proxy reads before it
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->w_empty[sw]);
            ++w_iter;
            const int st = a_iter % kNA;
            if (!mbar_wait(&ctl->a_empty[st], ((a_iter / kNA) & 1u) ^ 1u, abort, p.status)) return;
            uint8_t* tile = As + st * kAStage;
            if (valid) {
                const __half z = __ushort_as_half(cze);
                const __half2 z1024 = __half2half2(__hadd(__float2half_rn(1024.0f), z));
                const __half2 zneg = __half2half2(__hneg(__hadd(__float2half_rn(64.0f), z)));
                const __half2 sc = __half2half2(__ushort_as_half(csc));
                const uint32_t w[16] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w, cur[1].x, cur[1].y,
                                        cur[1].z, cur[1].w, cur[2].x, cur[2].y, cur[2].z, cur[2].w,
                                        cur[3].x, cur[3].y, cur[3].z, cur[3].w};
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint4 o = dequant8(w[j], z1024, zneg, sc);
                    const int k = j * 8;   // 0..120 within the group
                    *reinterpret_cast<uint4*>(tile + (k >> 6) * kASub + sw128_offset(r, k & 63)) = o;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int k = j * 8;
                    *reinterpret_cast<uint4*>(tile + (k >> 6) * kASub + sw128_offset(r, k & 63)) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->a_full[st]);
            ++a_iter;
            csc = nsc;
            cze = nze;
        }
    }
}

// ---- role: W3A16 GEMM producer (3-bit planes -> fp16 (q - z) * scale) ----
// Rotating plane p of a 32-level block right by (i - p) mod 32 puts bit i of
// the plane at bit p and bit i + 16 at bit 16 + p; OR-ing the three under
// the mantissa of fp16 1024 gives the exact pair (1024 + q_i, 1024 + q_{i+16}),
// and one HSUB2 the exact (q - z) pair.  Times the fp16 scale (HMUL2) it is
// rounded once to fp16, as in the 4-bit producer.  The pairs (i, i+16) of
// i = 8m .. 8m + 7 are then gathered (PRMT) into the 16-byte chunks of levels
// 8m .. 8m + 7 (low halves) and 16 + 8m .. (high halves).
__device__ __forceinline__ uint32_t rotr32(uint32_t w, uint32_t n) { return __funnelshift_r(w, w, n); }

__device__ __forceinline__ void dequant_block3(uint32_t p0, uint32_t p1, uint32_t p2,
                                               __half2 z1024, __half2 sc, uint4 (&o)[4]) {
    uint32_t pr[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t v = lop3_and_or(rotr32(p0, (uint32_t)i & 31u), 0x00010001u, 0x64006400u);
        v = lop3_and_or(rotr32(p1, (uint32_t)(i - 1) & 31u), 0x00020002u, v);
        v = lop3_and_or(rotr32(p2, (uint32_t)(i - 2) & 31u), 0x00040004u, v);
        pr[i] = h2u(__hmul2(__hsub2(u2h(v), z1024), sc));
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        o[m] = make_uint4(prmt(pr[8 * m], pr[8 * m + 1], 0x5410), prmt(pr[8 * m + 2], pr[8 * m + 3], 0x5410),
                          prmt(pr[8 * m + 4], pr[8 * m + 5], 0x5410), prmt(pr[8 * m + 6], pr[8 * m + 7], 0x5410));
        o[m + 2] = make_uint4(prmt(pr[8 * m], pr[8 * m + 1], 0x7632), prmt(pr[8 * m + 2], pr[8 * m + 3], 0x7632),
                              prmt(pr[8 * m + 4], pr[8 * m + 5], 0x7632), prmt(pr[8 * m + 6], pr[8 * m + 7], 0x7632));
    }
}

__device__ void role_prod_gemm3(const TcParams& p, uint8_t* As, SmemCtl* ctl, int r, int lane) {
    volatile int* abort = &ctl->abort;
    const int64_t wstride = p.K / 32 * 3;                // plane words per row
    uint32_t a_iter = 0;
    Item it;
    for (int li = 0; cta_item<kModeGemm3>(li, p, it); ++li) {
        const int64_t n = (int64_t)it.n_tile * kTcRows + r;
        const bool valid = n < p.N;
        const uint4* prow = reinterpret_cast<const uint4*>(p.planes + (valid ? n : 0) * wstride);
        const uint16_t* srow = p.scales + (valid ? n : 0) * p.G;
        const uint16_t* zrow = p.zeros + (valid ? n : 0) * p.G;
        uint4 cur[3];
        uint16_t csc = 0, cze = 0;
        if (valid) {
#pragma unroll
            for (int j = 0; j < 3; ++j) cur[j] = __ldg(prow + (int64_t)it.g0 * 3 + j);
            csc = __ldg(srow + it.g0);
            cze = __ldg(zrow + it.g0);
            for (int g = it.g0 + 2; g < it.g1 && g < it.g0 + kProdPrefetch; ++g)
                prefetch_l2(prow + (int64_t)g * 3);
        }
        for (int g = it.g0; g < it.g1; ++g) {
            uint4 nxt[3];
            uint16_t nsc = 0, nze = 0;
            if (valid && g + kProdPrefetch < it.g1) prefetch_l2(prow + (int64_t)(g + kProdPrefetch) * 3);
            if (valid && g + 1 < it.g1) {
#pragma unroll
                for (int j = 0; j < 3; ++j) nxt[j] = __ldg(prow + (int64_t)(g + 1) * 3 + j);
                nsc = __ldg(srow + g + 1);
                nze = __ldg(zrow + g + 1);
            }
            const int st = a_iter % kNA;
            if (!mbar_wait(&ctl->a_empty[st], ((a_iter / kNA) & 1u) ^ 1u, abort, p.status)) return;
            uint8_t* tile = As + st * kAStage;
            if (valid) {
                const __half2 z1024 =
                    __half2half2(__hadd(__float2half_rn(1024.0f), __ushort_as_half(cze)));
                const __half2 sc = __half2half2(__ushort_as_half(csc));
                const uint32_t w[12] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w, cur[1].x, cur[1].y,
                                        cur[1].z, cur[1].w, cur[2].x, cur[2].y, cur[2].z, cur[2].w};
#pragma unroll
                for (int b = 0; b < 4; ++b) {            // 32-level blocks of the group
                    uint4 o[4];
                    dequant_block3(w[3 * b], w[3 * b + 1], w[3 * b + 2], z1024, sc, o);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int k = 32 * b + 8 * m;    // 0..120 within the group
                        *reinterpret_cast<uint4*>(tile + (k >> 6) * kASub + sw128_offset(r, k & 63)) =
                            o[m];
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int k = j * 8;
                    *reinterpret_cast<uint4*>(tile + (k >> 6) * kASub + sw128_offset(r, k & 63)) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->a_full[st]);
            ++a_iter;
            if (valid && g + 1 < it.g1) {
#pragma unroll
                for (int j = 0; j < 3; ++j) cur[j] = nxt[j];
                csc = nsc;
                cze = nze;
            }
        }
    }
}

// ---- role: search producer (fake-quantise W diag(s), residual E in fp16) ----
// Four lanes hold one row of the group: lane c the 16-byte chunks c and c + 4
// of both 64-channel sub-tiles (channels 8c..8c+7, 32+8c.., 64+8c..,
// 96+8c..), 32 channels in all, so the group's range takes two shuffle
// rounds and each lane forms the group parameters once per 32 elements.  A
// warp covers 8 rows, the 16 producer warps the 128-row tile in one pass.
//
// The lane keeps -w' = -fp32(W s) (the fp16 sign flipped before the
// product, so exactly the negated product) as 16 pairs; the pair operations
// round each lane as the scalar ones do.  The levels are the packer's (same
// rounding points): with t = fp32(w' / d) by the fast exact quotient, the
// level offset (q - z) = rint(clamp(t, -z, qmax - z)) (clamping before or
// after rounding agree, the bounds being integers) is y - 1.5 * 2^23 with y =
// fp32(t + 1.5 * 2^23).  When rint(lo / d) and rint(hi / d) already fall in
// [-z, qmax - z] for every row of the warp, no t of the group leaves the
// range and the clamp is skipped.  A chunk whose quotient comes near a tie
// for any lane of the warp is redone with the exact quotient.
// E = (q - z) scale / s - W is formed as ((q - z) scale - w') (1/s): the FMA
// rounds (q - z) scale - w' once, and (q - z) scale is exact (at most 4 + 11
// significant bits), so this is the value of one fp32 subtraction; times 1/s
// and rounded to fp16.
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// -w' for the 8 channels of one 16-byte chunk of W, as 4 pairs.
__device__ __forceinline__ void unpack8_neg(uint4 v, float4 sa, float4 sb, float2* wn) {
    const uint32_t h[4] = {v.x ^ 0x80008000u, v.y ^ 0x80008000u, v.z ^ 0x80008000u,
                           v.w ^ 0x80008000u};
    const float2 s[4] = {make_float2(sa.x, sa.y), make_float2(sa.z, sa.w),
                         make_float2(sb.x, sb.y), make_float2(sb.z, sb.w)};
#pragma unroll
    for (int j = 0; j < 4; ++j)
        wn[j] = __fmul2_rn(__half22float2(*reinterpret_cast<const __half2*>(&h[j])), s[j]);
}

// The level offsets (q - z) of one chunk (4 pairs of -w'), and whether any
// of its quotients came near a tie.
template <bool CLAMP>
__device__ __forceinline__ bool chunk_levels(const float2* wn, float2 nrcp2, float lo_z, float hi_z,
                                             float2* rt) {
    const float kM = 12582912.0f;               // 1.5 * 2^23
    const float2 m2 = make_float2(kM, kM), negm2 = make_float2(-kM, -kM);
    const float2 neg1 = make_float2(-1.0f, -1.0f);
    float dm = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float2 t = __fmul2_rn(wn[j], nrcp2);    // (-w') (-1/d)
        if (CLAMP) {
            t.x = fminf(fmaxf(t.x, lo_z), hi_z);
            t.y = fminf(fmaxf(t.y, lo_z), hi_z);
        }
        rt[j] = __fadd2_rn(__fadd2_rn(t, m2), negm2);
        const float2 d = __ffma2_rn(rt[j], neg1, t);
        dm = fmax3_nan(dm, fabsf(d.x), fabsf(d.y));
    }
    return dm > kTieBand;
}

// The exact-quotient redo of one chunk: near-tie values take rint of the
// IEEE quotient, clamped.
__device__ __forceinline__ void chunk_levels_exact(const float2* wn, float scale, float rcp,
                                                   float lo_z, float hi_z, float2* rt) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float* r = reinterpret_cast<float*>(&rt[j]);
        const float* w = reinterpret_cast<const float*>(&wn[j]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float t = fminf(fmaxf(__fmul_rn(-w[h], rcp), lo_z), hi_z);
            if (near_tie(t, r[h]))
                r[h] = fminf(fmaxf(rintf(__fdiv_rn(-w[h], scale)), lo_z), hi_z);
        }
    }
}

template <int PW, bool GRAM>
__device__ void role_prod_search(const TcParams& p, uint8_t* As, SmemCtl* ctl, int pw, int lane) {
    static_assert(PW * 8 == kTcRows, "16 producer warps x 8 rows");
    volatile int* abort = &ctl->abort;
    const int rr = lane >> 2, c = lane & 3;
    const int r = pw * 8 + rr;                          // this lane's row of the tile
    // the lane's four chunks q: sub-tile q / 2, chunk c + 4 (q % 2) (k = 64 (q / 2) + 8 c
    // + 32 (q % 2)); within a sub-tile the two chunks sit 64 bytes apart after the
    // swizzle (chunk index XOR row % 8 flips only its low three bits)
    const uint32_t soff0 = sw128_offset(r, 8 * c);
    uint32_t a_iter = 0, item_iter = 0;
    bool bad = false;
    Item it;
    for (int li = 0; cta_item<kModeSearch>(li, p, it); ++li, ++item_iter) {
        // Gram route: the groups of this item's 512 output columns, whose
        // residuals the epilogue needs (exported into this CTA's buffer
        // item_iter % 2, [128 rows][512 columns] fp16)
        const int g_par = it.t_tile * 4;
        uint16_t* e_row = GRAM ? p.e_exp +
                                     ((int64_t)(blockIdx.x * 2 + (item_iter & 1)) * kTcRows + r) *
                                         kSearchTokensPerItem
                               : nullptr;
        if (GRAM && !mbar_wait(&ctl->par_empty[item_iter & 1], ((item_iter >> 1) & 1u) ^ 1u, abort,
                               p.status))
            return;
        const float* s_a = p.s_alpha + (int64_t)it.alpha * p.K;
        const float* is_a = p.inv_s_alpha + (int64_t)it.alpha * p.K;
        const int64_t n = (int64_t)it.n_tile * kTcRows + r;
        const bool valid = n < p.N;
        const uint16_t* wrow = p.W + (valid ? n : 0) * p.ldw;
        for (int g = 0; g < p.G; ++g) {
            const int64_t kg = (int64_t)g * kGroup;
            uint4 raw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = 64 * (q >> 1) + 8 * (c + 4 * (q & 1));
                raw[q] = valid ? __ldg(reinterpret_cast<const uint4*>(wrow + kg + k))
                               : make_uint4(0, 0, 0, 0);
            }
            // phase 1: -w' for the 32 channels, and the range of w'
            float2 wn[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = 64 * (q >> 1) + 8 * (c + 4 * (q & 1));
                const float4* sp = reinterpret_cast<const float4*>(s_a + kg + k);
                unpack8_neg(raw[q], __ldg(sp), __ldg(sp + 1), wn + 4 * q);
            }
            float mn[4], mx[4];                 // four independent chains over -w'
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                mn[q] = fmin_nan(wn[q].x, wn[q].y);
                mx[q] = fmax_nan(wn[q].x, wn[q].y);
            }
#pragma unroll
            for (int e = 4; e < 16; ++e) {
                mn[e & 3] = fmin3_nan(mn[e & 3], wn[e].x, wn[e].y);
                mx[e & 3] = fmax3_nan(mx[e & 3], wn[e].x, wn[e].y);
            }
            float lo = -fmax_nan(fmax3_nan(mx[0], mx[1], mx[2]), mx[3]);
            float hi = -fmin_nan(fmin3_nan(mn[0], mn[1], mn[2]), mn[3]);
            // this lane's 32 values: NaN or Inf makes lo or hi non-finite
            bad |= !(isfinite(lo) && isfinite(hi));
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
            }
            const GroupQuant gq = group_quant_from_range(lo, hi, p.qmax);
            bad |= !gq.finite;
            const float lo_z = -gq.zf, hi_z = p.qmax - gq.zf;
            const bool inside = __all_sync(0xffffffffu,
                                           rint_small(__fmul_rn(lo, gq.rcp)) >= lo_z &&
                                               rint_small(__fmul_rn(hi, gq.rcp)) <= hi_z);
            const float2 nrcp2 = make_float2(-gq.rcp, -gq.rcp), sc2 = make_float2(gq.scale, gq.scale);
            const int st = a_iter % kNA;
            if (!mbar_wait(&ctl->a_empty[st], ((a_iter / kNA) & 1u) ^ 1u, abort, p.status)) return;
            uint8_t* tile = As + st * kAStage;
            // phase 2: levels, residual, fp16, one 16-byte store per chunk
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = 64 * (q >> 1) + 8 * (c + 4 * (q & 1));
                const float4 i0 = __ldg(reinterpret_cast<const float4*>(is_a + kg + k));
                const float4 i1 = __ldg(reinterpret_cast<const float4*>(is_a + kg + k + 4));
                const float2 is2[4] = {make_float2(i0.x, i0.y), make_float2(i0.z, i0.w),
                                       make_float2(i1.x, i1.y), make_float2(i1.z, i1.w)};
                float2 rt[4];
                const bool tie = inside ? chunk_levels<false>(wn + 4 * q, nrcp2, lo_z, hi_z, rt)
                                        : chunk_levels<true>(wn + 4 * q, nrcp2, lo_z, hi_z, rt);
                if (__any_sync(0xffffffffu, tie))
                    chunk_levels_exact(wn + 4 * q, gq.scale, gq.rcp, lo_z, hi_z, rt);
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 ev = __fmul2_rn(__ffma2_rn(rt[j], sc2, wn[4 * q + j]), is2[j]);
                    o[j] = pack_h2(ev.x, ev.y);
                }
                const uint32_t off = (uint32_t)((q >> 1) * kASub) + ((q & 1) ? (soff0 ^ 64u) : soff0);
                *reinterpret_cast<uint4*>(tile + off) = make_uint4(o[0], o[1], o[2], o[3]);
                if (GRAM && g >= g_par && g < g_par + 4)
                    *reinterpret_cast<uint4*>(e_row + (g - g_par) * kGroup + k) =
                        make_uint4(o[0], o[1], o[2], o[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->a_full[st]);
            ++a_iter;
        }
        if (GRAM) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->par_full[item_iter & 1]);
        }
    }
    if (bad) set_status(p.status, kStatusNonFinite);
}

template <int MODE>
__global__ void __launch_bounds__(Cfg<MODE>::kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapA,
              const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* As = smem;
    uint8_t* Bs = smem + kNA * kAStage;
    uint8_t* Ws = Bs + kNB * kBStage;                   // GEMM: packed-word ring
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(Ws + ring_w_bytes<MODE>());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNA; ++i) {
            // the A stages are filled by the producer warps, or by TMA (X^T X)
            mbar_init(&ctl->a_full[i], Cfg<MODE>::kProdWarps > 0 ? Cfg<MODE>::kProdWarps : 1);
            mbar_init(&ctl->a_empty[i], 1);
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(&ctl->b_full[i], 1);
            mbar_init(&ctl->b_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->acc_full[i], 1);
            mbar_init(&ctl->acc_empty[i], 4);
            mbar_init(&ctl->par_full[i], Cfg<MODE>::kProdWarps > 0 ? Cfg<MODE>::kProdWarps : 1);
            mbar_init(&ctl->par_empty[i], 4);
        }
        for (int i = 0; i < kNW; ++i) {
            mbar_init(&ctl->w_full[i], 1);
            mbar_init(&ctl->w_empty[i], Cfg<MODE>::kProdWarps > 0 ? Cfg<MODE>::kProdWarps : 1);
        }
        mbar_init(&ctl->mma_done, 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == kWarpTmem) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&mapX);
        if (MODE == kModeXtX || MODE == kModeGemm) tma_prefetch_desc(&mapA);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    // Launched as a programmatic dependent: the set-up above overlapped the
    // previous kernel; every role waits for its writes here, except the
    // weight producers of a GEMM whose previous kernel writes no weights.
    if (!(is_gemm<MODE>() && p.early_w &&
          (warp >= kWarpProd0 || (MODE == kModeGemm && warp == kWarpTmaW))))
        grid_dep_wait();

    if (warp == kWarpTma) {
        if (lane == 0) role_tma<MODE>(&mapX, &mapA, p, As, Bs, ctl);
    } else if (warp == kWarpMma) {
        if (lane == 0) role_mma<MODE>(p, As, Bs, ctl, tmem);
    } else if (MODE == kModeGemm && warp == kWarpTmaW) {
        if (lane == 0) role_tma_w(&mapA, p, Ws, ctl);
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
        role_epilogue<MODE>(p, ctl, tmem, warp - kWarpEpi0, lane);
    } else if (warp >= kWarpProd0) {
        if constexpr (MODE == kModeGemm)
            role_prod_gemm(p, As, Ws, ctl, (warp - kWarpProd0) * 32 + lane, lane);
        else if constexpr (MODE == kModeGemm3)
            role_prod_gemm3(p, As, ctl, (warp - kWarpProd0) * 32 + lane, lane);
        else if constexpr (MODE == kModeSearch)
            role_prod_search<Cfg<MODE>::kProdWarps, false>(p, As, ctl, warp - kWarpProd0, lane);
        else if constexpr (MODE == kModeGram)
            role_prod_search<Cfg<MODE>::kProdWarps, true>(p, As, ctl, warp - kWarpProd0, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpTmem) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int MODE>
cudaError_t launch_tc(const CUtensorMap& mapX, const CUtensorMap& mapA, const TcParams& p,
                      int num_sms, cudaStream_t st) {
    if (p.n_items <= 0) return cudaSuccess;
    constexpr size_t kSmem = smem_bytes<MODE>();
    cudaError_t e = smem_attr_once<tc_kernel<MODE>>((int)kSmem);
    if (e != cudaSuccess) return e;
    const int grid = p.n_items < num_sms ? p.n_items : num_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Cfg<MODE>::kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_kernel<MODE>, mapX, mapA, p);
}

__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float* __restrict__ ws, int k_splits, int64_t M, int64_t N,
                         uint16_t* __restrict__ Y, int64_t ldy) {
    const int64_t per = M * N;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per; i += stride) {
        float acc = ws[i];
        for (int s = 1; s < k_splits; ++s) acc += ws[(int64_t)s * per + i];
        const int64_t m = i / N, n = i - m * N;
        Y[m * ldy + n] = __half_as_ushort(__float2half_rn(acc));
    }
}

// The stream-K tail's fixup: block (x, t) adds, for tail tile t, 1024
// consecutive elements (4 per thread, [token][row] order) of the tile's
// partial slots in CTA order (ascending groups) and rounds them to fp16 into
// Y.  It is launched as a programmatic dependent of the GEMM: the slot list,
// which depends only on the schedule, is formed (by one warp, 32 CTAs at a
// time) while the GEMM's last CTAs finish, and the partials are read after
// griddepcontrol.wait.  NF slots' loads are issued together and the adds
// stay in slot order; a wider batch takes more registers, hence fewer blocks
// per SM (the launcher picks NF from the slots per tile and the block count).
constexpr int kSkFixThreads = 256;
constexpr int kSkFixElems = 4 * kSkFixThreads;
constexpr int kSkMaxSlots = 512;

template <int NF>
constexpr int sk_fix_blocks_per_sm() {
    return NF >= 16 ? 2 : NF >= 8 ? 4 : 5;
}

template <int NF>
__global__ void __launch_bounds__(kSkFixThreads, sk_fix_blocks_per_sm<NF>())
    sk_fixup_kernel(const TcParams p) {
    constexpr int kTileElems = kTcRows * kTcTokens;
    __shared__ int slots[kSkMaxSlots];
    __shared__ int n_slots;
    const int t = blockIdx.y;
    if (threadIdx.x < 32) {
        // the CTAs whose shares meet units [t G, (t + 1) G): c(u) is the CTA
        // with s_c <= u < s_(c+1); those with empty shares are left out
        const int lane = threadIdx.x;
        const int64_t units = (int64_t)p.sk_tiles * p.G;
        const int64_t u0 = (int64_t)t * p.G, u1 = u0 + p.G - 1;
        const int c0 = (int)(((u0 + 1) * p.sk_ctas + units - 1) / units) - 1;
        const int c1 = (int)(((u1 + 1) * p.sk_ctas + units - 1) / units) - 1;
        int k = 0;
        for (int cb = c0; cb <= c1; cb += 32) {
            const int c = cb + lane;
            int64_t s0 = 0, s1 = 0;
            if (c <= c1) sk_share(c, p.sk_ctas, p.sk_tiles, p.G, s0, s1);
            const bool has = c <= c1 && s0 < s1;
            const unsigned m = __ballot_sync(0xffffffffu, has);
            const int pos = k + __popc(m & ((1u << lane) - 1u));
            if (has && pos < kSkMaxSlots) slots[pos] = 2 * c + (s0 / p.G == t ? 0 : 1);
            k += __popc(m);
        }
        if (lane == 0) n_slots = k < kSkMaxSlots ? k : kSkMaxSlots;
    }
    __syncthreads();
    const Item it = decode_item<kModeGemm>(p.sk_full + t, p);
    const int off = blockIdx.x * kSkFixElems + 4 * threadIdx.x;      // token * 128 + row
    const int64_t n = (int64_t)it.n_tile * kTcRows + (off % kTcRows);
    const int64_t tok = (int64_t)it.t_tile * kTcTokens + off / kTcRows;
    if (tok >= p.rows_tok) return;
    grid_dep_wait();
    const int ns = n_slots;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* base = p.ws_sk + off;
    for (int k = 0; k < ns; k += NF) {
        float4 v[NF];
#pragma unroll
        for (int u = 0; u < NF; ++u)
            if (k + u < ns)
                v[u] = __ldcs(reinterpret_cast<const float4*>(base + (int64_t)slots[k + u] * kTileElems));
#pragma unroll
        for (int u = 0; u < NF; ++u) {
            if (k + u < ns) {
                acc.x += v[u].x;
                acc.y += v[u].y;
                acc.z += v[u].z;
                acc.w += v[u].w;
            }
        }
    }
    unsigned short* y = reinterpret_cast<unsigned short*>(p.Y) + tok * p.ldy + n;
    const float a[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if (n + e < p.N) y[e] = __half_as_ushort(__float2half_rn(a[e]));
}

}  // namespace

cudaError_t launch_sk_fixup(const TcParams& p, cudaStream_t st) {
    if (p.sk_tiles <= 0) return cudaSuccess;
    // a tile's shares come from at most 2 sk_ctas CTAs (one or two pieces each)
    if (2 * p.sk_ctas > kSkMaxSlots) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kTcRows * kTcTokens / kSkFixElems, (unsigned)p.sk_tiles);
    cfg.blockDim = dim3(kSkFixThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the batch width with the fewest (waves of blocks) x (load rounds): a
    // tile meets at most ceil(sk_ctas / sk_tiles) + 1 shares
    int num_sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        num_sms = p.sk_ctas;
    const int64_t blocks = (int64_t)cfg.gridDim.x * cfg.gridDim.y;
    const int slots = (p.sk_ctas + p.sk_tiles - 1) / p.sk_tiles + 1;
    auto cost = [&](int nf, int per_sm) {
        const int64_t conc = (int64_t)num_sms * per_sm;
        return ((blocks + conc - 1) / conc) * (int64_t)((slots + nf - 1) / nf);
    };
    const int64_t c16 = cost(16, sk_fix_blocks_per_sm<16>());
    const int64_t c8 = cost(8, sk_fix_blocks_per_sm<8>());
    const int64_t c4 = cost(4, sk_fix_blocks_per_sm<4>());
    if (c16 < c8 && c16 < c4) return cudaLaunchKernelEx(&cfg, sk_fixup_kernel<16>, p);
    if (c8 < c4) return cudaLaunchKernelEx(&cfg, sk_fixup_kernel<8>, p);
    return cudaLaunchKernelEx(&cfg, sk_fixup_kernel<4>, p);
}

cudaError_t launch_splitk_reduce(const float* ws_partial, int k_splits, int64_t M, int64_t N,
                                 uint16_t* Y, int64_t ldy, int num_sms, cudaStream_t st) {
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, st>>>(ws_partial, k_splits, M, N, Y, ldy);
    return cudaGetLastError();
}

cudaError_t launch_tc_gemm(const CUtensorMap& mapX, const CUtensorMap& mapW, const TcParams& p,
                           int num_sms, cudaStream_t st) {
    return launch_tc<kModeGemm>(mapX, mapW, p, num_sms, st);
}
cudaError_t launch_tc_search(const CUtensorMap& mapX, const TcParams& p, int num_sms,
                             cudaStream_t st) {
    return launch_tc<kModeSearch>(mapX, mapX, p, num_sms, st);
}
cudaError_t launch_tc_gemm3(const CUtensorMap& mapX, const TcParams& p, int num_sms,
                            cudaStream_t st) {
    return launch_tc<kModeGemm3>(mapX, mapX, p, num_sms, st);
}
cudaError_t launch_tc_xtx(const CUtensorMap& mapB, const CUtensorMap& mapA, const TcParams& p,
                          int num_sms, cudaStream_t st) {
    return launch_tc<kModeXtX>(mapB, mapA, p, num_sms, st);
}
cudaError_t launch_tc_gram_search(const CUtensorMap& mapG, const TcParams& p, int num_sms,
                                  cudaStream_t st) {
    return launch_tc<kModeGram>(mapG, mapG, p, num_sms, st);
}

}  // namespace awq
