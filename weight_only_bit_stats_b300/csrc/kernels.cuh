// Host-side launchers of the library's kernels (private to the library).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace awq {

struct AlphaList {
    double a[64];
};

// ---- statistics (stats.cu) ----
cudaError_t launch_act_stats(const uint16_t* X, int64_t T, int64_t K, int64_t ldx,
                             unsigned long long* abs_sum, unsigned* status, int num_sms,
                             cudaStream_t st);
cudaError_t launch_act_mean(const int64_t* abs_sum, int64_t n_tokens, int64_t K, double* mean,
                            cudaStream_t st);

// Diagnostic: a bounded wait on an mbarrier nothing arrives on (stats.cu).
cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, unsigned* status,
                                         cudaStream_t st);

// ---- candidate scales, pack, search reduction (quant.cu) ----
int cand_blocks(int64_t K);
// ws_r: [n_alpha, K] fp64; ws_mm: [n_alpha, cand_blocks(K), 2] fp64.
cudaError_t launch_candidate_scales(const double* mean, int64_t K, const AlphaList& alphas,
                                    int n_alpha, float* s_alpha, float* inv_s_alpha, double* ws_r,
                                    double* ws_mm, cudaStream_t st);
cudaError_t launch_pack_int4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw, const float* s,
                             uint32_t* qweight, uint16_t* scales, uint16_t* zeros, unsigned* status,
                             int num_sms, cudaStream_t st);
// mse[a] = sum_i partials[a][i] / (T N) for i < n_part; best = first argmin;
// s_out = s_alpha[best].
cudaError_t launch_search_finalize(const double* partials, int n_alpha, int64_t n_part, int64_t T,
                                   int64_t N, int64_t K, const float* s_alpha, double* mse,
                                   int32_t* best_idx, float* s_out, cudaStream_t st);

// ---- decode matmul, M <= 16 (gemv.cu) ----
struct GemvParams {
    const uint16_t* X;
    int64_t ldx;
    int M;
    const uint32_t* qw;
    const uint16_t* scales;
    const uint16_t* zeros;
    int64_t N, K;
    int G;
    uint16_t* Y;
    int64_t ldy;
    unsigned* status;
    int early_weights;   // 1: weights may be fetched before the previous kernel completes
    const float* inv_s;  // [K] or null: X is used as fp16(X * inv_s) (fused input scaling)
};
// mapW: 2-D tensor map of qweight as uint32 [N rows][K/8 words], box 48 words x 16 rows.
cudaError_t launch_gemv(const CUtensorMap& mapW, const GemvParams& p, int num_sms,
                        cudaStream_t st);

// ---- decode matmul over the repacked decode tiles, and the repack
// (gemv_tiles.cu) ----
constexpr int kTileBytes = 1088;   // one (16-row slab, group of 128) tile, 4 bits
constexpr int kTile3Bytes = 832;   // the same at 3 bits: 16 x 48 bytes of planes + 64
struct TileParams {
    const uint16_t* X;
    int64_t ldx;
    int M;
    const uint8_t* tiles;   // ceil(N / 16) * G tiles of kTileBytes
    int64_t N;
    int G;
    uint16_t* Y;
    int64_t ldy;
    unsigned* status;
    int early_weights;   // 1: weights may be fetched before the previous kernel completes
    const float* inv_s;  // [K] or null: X is used as fp16(X * inv_s) (4 bits only)
    int bits;            // 4 or 3 (tiles of kTileBytes or kTile3Bytes)
};
cudaError_t launch_gemv_tiles(const TileParams& p, int num_sms, cudaStream_t st);
cudaError_t launch_repack_int3(const uint32_t* planes, const uint16_t* scales,
                               const uint16_t* zeros, int64_t N, int64_t K, void* tiles,
                               int num_sms, cudaStream_t st);
cudaError_t launch_repack_int4(const uint32_t* qweight, const uint16_t* scales,
                               const uint16_t* zeros, int64_t N, int64_t K, void* tiles,
                               int num_sms, cudaStream_t st);

// ---- tensor-core kernels (tc.cu): W4A16 GEMM and the alpha search ----
struct TcParams {
    int N, K, G;
    int rows_tok;    // M (GEMM) or T (search): rows of the TMA-loaded activations
    int n_tiles;     // ceil(N / 128)
    int t_tiles;     // ceil(rows_tok / tokens per item)
    int n_items;
    // GEMM
    const uint32_t* qw;
    const uint16_t* scales;
    const uint16_t* zeros;
    uint16_t* Y;
    int64_t ldy;
    int k_splits;          // K split over this many items per output tile (1: none)
    float* ws_partial;     // k_splits > 1: fp32 partials [k_splits][rows_tok][N]
    // search
    const uint16_t* W;
    int64_t ldw;
    const float* s_alpha;
    const float* inv_s_alpha;
    int n_alpha;
    double* partials;  // [n_alpha][n_tiles][t_tiles][4]
    unsigned* status;
    // X^T X: fp16 out [N][rows_tok] (= [K][K]) scaled by inv_t
    uint16_t* gout;
    float inv_t;
    // search: top quantisation level (15 at 4 bits, 7 at 3 bits)
    float qmax;
    // 3-bit GEMM: bit planes [N][K/32][3] in place of qw
    const uint32_t* planes;
    // Gram-route search: per CTA two [128][512] fp16 buffers through which
    // the producer hands the epilogue the residuals of an item's columns
    uint16_t* e_exp;
    // GEMM modes: the weight producers may read qw / planes, scales and
    // zeros before the previous kernel in the stream has completed (that
    // kernel writes none of them)
    int early_w;
    // GEMM stream-K tail (k_splits == 1, sk_tiles > 0): the first sk_full
    // output tiles (a multiple of sk_ctas) run whole, one per CTA in turn;
    // the K range of the last sk_tiles tiles is cut into sk_ctas equal
    // shares of groups, one per CTA, each written as fp32 partial tiles
    // (slots 2c, 2c + 1 of CTA c, [256 tokens][128 rows]) to ws_sk and
    // added by launch_sk_fixup.  The grid is sk_ctas CTAs.
    int sk_full, sk_tiles, sk_ctas;
    float* ws_sk;
};
constexpr int kTcRows = 128;          // weight rows per tile (UMMA M)
constexpr int kTcTokens = 256;        // tokens per accumulator slot (UMMA N)
constexpr int kGemmTokensPerItem = 256;
constexpr int kSearchTokensPerItem = 512;

// mapX: the activations [M, K] fp16; mapW: qweight [N, K/8] uint32 in boxes
// of one group x 128 rows, 64-byte swizzle.
cudaError_t launch_tc_gemm(const CUtensorMap& mapX, const CUtensorMap& mapW, const TcParams& p,
                           int num_sms, cudaStream_t st);
// inv[i] = fp32(1 / s[i]), correctly rounded, for n values.
cudaError_t launch_reciprocals(const float* s, int64_t n, float* inv, int num_sms,
                               cudaStream_t st);
// Xs[m, k] = fp16(fp32(X[m, k]) * inv_s[k]) into a dense [M, K] buffer.
cudaError_t launch_scale_x(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                           const float* inv_s, uint16_t* Xs, int num_sms, cudaStream_t st);
// The stream-K tail's output tiles: Y = fp16(sum of each tile's partial
// slots in CTA order).
cudaError_t launch_sk_fixup(const TcParams& p, cudaStream_t st);
// Y = fp16(sum over splits of ws_partial), the splits added in order.
cudaError_t launch_splitk_reduce(const float* ws_partial, int k_splits, int64_t M, int64_t N,
                                 uint16_t* Y, int64_t ldy, int num_sms, cudaStream_t st);
cudaError_t launch_tc_search(const CUtensorMap& mapX, const TcParams& p, int num_sms,
                             cudaStream_t st);
// G/T = X^T X / T into p.gout: both operands are tiles of X^T [K][T_pad]
// (mapB: boxes of 64 x 256 rows, mapA: 64 x 128 rows).  p.N = p.rows_tok = K.
cudaError_t launch_tc_xtx(const CUtensorMap& mapB, const CUtensorMap& mapA, const TcParams& p,
                          int num_sms, cudaStream_t st);
// The alpha search through G/T (mapG: G/T [K][K] fp16, boxes of 64 x 256
// rows); partials as the direct search, already divided by T.
cudaError_t launch_tc_gram_search(const CUtensorMap& mapG, const TcParams& p, int num_sms,
                                  cudaStream_t st);
// W3A16 GEMM for M > 16 over the 3-bit planes (p.planes, p.scales, p.zeros);
// no split-K (k_splits must be 1).
cudaError_t launch_tc_gemm3(const CUtensorMap& mapX, const TcParams& p, int num_sms,
                            cudaStream_t st);
// X^T [K][T_pad] (zero columns past T) from X [T][K] (leading dimension ldx).
cudaError_t launch_transpose_x(const uint16_t* X, int64_t T, int64_t K, int64_t ldx,
                               uint16_t* Xt, int64_t T_pad, cudaStream_t st);

}  // namespace awq
