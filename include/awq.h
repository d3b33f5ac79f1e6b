/*
 * awq.h -- C ABI of the B300 (sm_103a) AWQ hot-path library libawq_b300.so.
 *
 * The method: "AWQ: Activation-aware Weight Quantization for On-Device LLM
 * Compression and Acceleration" (fdeinterviews.com/papers/awq).  Third
 * paragraph: scaling a weight channel up by s > 1 and its input down by the
 * same factor keeps the layer's output while lowering that channel's
 * relative rounding error; s is a power alpha of the channel's mean absolute
 * activation, alpha is picked by trying a small grid of values on a few
 * calibration samples, and all stored weights are low-bit.  Seventh
 * paragraph: the method gathers activation statistics and fits nothing.  First paragraph: decoding reads
 * every weight once per step and is memory-bound, so 4-bit weights cut its
 * traffic about 4x.  The OpenAlex record of the same title (abstract):
 * on-the-fly dequantisation and kernel fusion in the inference kernels.
 * Group size 128, asymmetric levels 0..15 with fp16 scale and zero-point,
 * mean |x| as the magnitude and output MSE as the search objective are this
 * library's stated workload definition; the pages leave them open.
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers owned by the caller unless stated
 *    otherwise.  The library never allocates device memory; scratch comes from
 *    a caller-provided workspace of at least the size its *_workspace_size()
 *    function returns (16-byte aligned).
 *  - fp16 data is passed as uint16_t bit patterns (IEEE binary16), so this
 *    header needs no CUDA header.  Matrices are row-major with the stated
 *    leading dimension (elements).
 *  - Calls are asynchronous and stream-ordered on `stream` (NULL = legacy
 *    default stream).  Host-side argument errors are returned immediately and
 *    nothing is launched.  Conditions found on the device (non-finite input,
 *    a bounded wait that expired) are recorded in a library status word on
 *    the current device; awq_sync_status() synchronises the stream and
 *    returns and clears it.
 *  - Calls that share a workspace race if they overlap on the GPU.
 *  - Requires a compute capability 10.3 device (B300); others get
 *    AWQ_ERR_DEVICE.
 */
#ifndef AWQ_B300_H
#define AWQ_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int awq_status;
enum {
    AWQ_OK = 0,
    AWQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad flag */
    AWQ_ERR_SHAPE = 2,       /* K % 128 != 0, group != 128, N % 8 != 0, ld < K */
    AWQ_ERR_ALIGN = 3,       /* pointer not 16-byte aligned or ld not a multiple of 8 */
    AWQ_ERR_DEVICE = 4,      /* current device is not sm_103 / no kernel image */
    AWQ_ERR_WORKSPACE = 5,   /* workspace missing or too small */
    AWQ_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
    AWQ_ERR_TIMEOUT = 7,     /* a bounded device-side wait expired */
    AWQ_ERR_NONFINITE = 8,   /* NaN/Inf input, or a group scale overflowing fp16 */
    AWQ_ERR_OVERFLOW = 9     /* an accumulated statistics sum left the exact int64 range */
};

/* Same type as cudaStream_t. */
typedef struct CUstream_st* awq_stream_t;

#define AWQ_GROUP 128
#define AWQ_MAX_ALPHAS 64

/* ---- step: calibration statistics ---------------------------------------
 * Per-input-channel sum of |x| over calibration tokens (the pages' "average
 * activation magnitude", third paragraph; statistics only, seventh paragraph).
 *   X            [T, K] fp16, leading dimension ldx (>= K, multiple of 8),
 *                16-byte aligned; K % 8 == 0.
 *   accumulate   0: abs_sum_q24 is overwritten; 1: this batch is added to
 *                it (stream calibration batches through one buffer).
 *   abs_sum_q24  [K] int64: sum_t |X[t,k]| * 2^24.  Every finite fp16 is an
 *                integer multiple of 2^-24 below 2^16, so the sums are exact
 *                integers and independent of summation order
 *                (bit-reproducible) while the running total stays below 2^63,
 *                which any 2^23 - 1 tokens guarantee.
 * T must be below 2^23 (AWQ_ERR_SHAPE otherwise).  With accumulate = 1 the
 * caller keeps the total token count of all batches below 2^23 for the same
 * guarantee; a running total that reaches 2^63 anyway flags AWQ_ERR_OVERFLOW
 * in the status word (the sums are then invalid).
 * NaN/Inf inputs are skipped and flag AWQ_ERR_NONFINITE in the status word. */
awq_status awq_act_stats(const uint16_t* X, int64_t T, int64_t K, int64_t ldx,
                         int accumulate, int64_t* abs_sum_q24, awq_stream_t stream);

/* mean_abs[k] = abs_sum_q24[k] / 2^24 / n_tokens (two IEEE fp64 divisions).
 *   abs_sum_q24 [K] int64 (device), mean_abs [K] fp64 (device), n_tokens > 0. */
awq_status awq_act_mean(const int64_t* abs_sum_q24, int64_t n_tokens, int64_t K,
                        double* mean_abs, awq_stream_t stream);

/* ---- step: candidate scales ---------------------------------------------
 * s = mean|x|^alpha, normalised (third paragraph).  For each alpha_i:
 *   r_k = pow(max(mean_abs[k], 1e-4), alpha_i)          (fp64)
 *   s_alpha[i*K + k] = fp32( r_k / sqrt(max_j r_j * min_j r_j) )
 * The normaliser only centres s around 1: a constant factor on s leaves the
 * quantised layer's output unchanged.
 *   mean_abs  [K] fp64 device.   alphas: HOST array of n_alpha fp64,
 *   1 <= n_alpha <= AWQ_MAX_ALPHAS.   s_alpha [n_alpha, K] fp32 device.
 *   workspace >= awq_candidate_scales_workspace_size(K, n_alpha) bytes. */
awq_status awq_candidate_scales(const double* mean_abs, int64_t K, const double* alphas,
                                int n_alpha, float* s_alpha, void* workspace,
                                size_t ws_bytes, awq_stream_t stream);
size_t awq_candidate_scales_workspace_size(int64_t K, int n_alpha);

/* ---- step: alpha grid search ---------------------------------------------
 * For every alpha on the grid (third paragraph: alpha is searched on a few
 * calibration samples, with no gradients and no refitting of weights):
 *   s = candidate scales (above); fake-quantise W diag(s) exactly as
 *   awq_pack_int4 does; E = Q(W diag(s)) diag(s)^-1 - W;
 *   mse(alpha) = ||Xcal E^T||_F^2 / (T N), the output MSE of
 *   Q(W diag(s)) diag(s)^-1 Xcal against W Xcal.
 * The best alpha is the smallest index with the least mse (ascending scan,
 * strict <).  Xcal E^T runs on the tensor cores (fp16 E, fp32 accumulation).
 *   W        [N, K] fp16, leading dimension ldw (>= K, multiple of 8).
 *   Xcal     [T, K] fp16, leading dimension ldx (>= K, multiple of 8).
 *   mean_abs [K] fp64 from awq_act_mean.
 *   alphas   HOST array of n_alpha fp64, 1 <= n_alpha <= AWQ_MAX_ALPHAS.
 *   group    must be 128.
 *   s_out    [K] fp32: s at the best alpha.
 *   mse_out  [n_alpha] fp64, may be NULL.
 *   best_idx [1] int32.
 *   s_alpha_out [n_alpha, K] fp32, may be NULL (all candidates, for checks).
 * K % 128 == 0, N % 8 == 0, T >= 1.  Pointers 16-byte aligned.
 * workspace >= awq_search_workspace_size(N, K, T, n_alpha) bytes. */
awq_status awq_search_scale(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                            const uint16_t* Xcal, int64_t T, int64_t ldx,
                            const double* mean_abs, const double* alphas, int n_alpha,
                            int group, float* s_out, double* mse_out, int32_t* best_idx,
                            float* s_alpha_out, void* workspace, size_t ws_bytes,
                            awq_stream_t stream);
size_t awq_search_workspace_size(int64_t N, int64_t K, int64_t T, int n_alpha);

/* The search step alone, on caller-given candidate scales (the grid search
 * of the third paragraph over any set of candidates): for each row a of
 * s_alpha, mse[a] and the first argmin exactly as awq_search_scale computes
 * them after its candidate step, with 1/s formed as fp32(1 / s) correctly
 * rounded (the candidate step's rule), so candidates from
 * awq_candidate_scales give awq_search_scale's results bit for bit.
 *   s_alpha  [n_alpha, K] fp32 device, 16-byte aligned, each s > 0.
 *   s_out    [K] fp32: the row of s_alpha at the best index.
 * Other arguments as awq_search_scale (4 bits); workspace >=
 * awq_search_mse_workspace_size(N, K, T, n_alpha) bytes. */
awq_status awq_search_mse(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                          const uint16_t* Xcal, int64_t T, int64_t ldx, const float* s_alpha,
                          int n_alpha, int group, float* s_out, double* mse_out,
                          int32_t* best_idx, void* workspace, size_t ws_bytes,
                          awq_stream_t stream);
size_t awq_search_mse_workspace_size(int64_t N, int64_t K, int64_t T, int n_alpha);

/* The same search at 3 bits (the pages evaluate 3 and 4 bits, fourth
 * paragraph): the fake quantiser is awq_pack_int3's (levels 0..7, scale =
 * fp16_rn(max(fp32(range / 7), 2^-14)), zero-point clamped to 0..7).
 * Arguments, results and workspace as awq_search_scale. */
awq_status awq_search_scale_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                 const uint16_t* Xcal, int64_t T, int64_t ldx,
                                 const double* mean_abs, const double* alphas, int n_alpha,
                                 int group, float* s_out, double* mse_out, int32_t* best_idx,
                                 float* s_alpha_out, void* workspace, size_t ws_bytes,
                                 awq_stream_t stream);

/* ---- alpha search through the Gram matrix ---------------------------------
 * The third paragraph picks alpha by a grid search on a few calibration
 * samples: that fixes the objective, not how it is evaluated.  ||Xcal E^T||_F^2 =
 * tr(E G E^T) with G = Xcal^T Xcal, so once G is formed the per-alpha cost is
 * 2 N K^2 flops instead of 2 T N K: cheaper whenever T > K (a full
 * calibration set of 128 x 512 tokens).
 *
 * awq_gram: G/T = Xcal^T Xcal / T as fp16 [K, K] (row-major, symmetric).
 * Each element is the fp32 tensor-core sum over the T tokens, times fp32(1/T),
 * rounded once to fp16.
 *   Xcal  [T, K] fp16, leading dimension ldx (>= K, multiple of 8).
 *   G     [K, K] fp16 out, 16-byte aligned.
 *   workspace >= awq_gram_workspace_size(T, K) bytes (a transposed copy of
 *   Xcal).  K % 128 == 0, T >= 1. */
size_t awq_gram_workspace_size(int64_t T, int64_t K);
awq_status awq_gram(const uint16_t* Xcal, int64_t T, int64_t K, int64_t ldx, uint16_t* G,
                    void* workspace, size_t ws_bytes, awq_stream_t stream);

/* awq_search_scale_gram: the alpha search of awq_search_scale with the
 * objective evaluated as
 *   mse(alpha) = sum_n (E G/T E^T)_nn / N,
 * E the same fp16 residual the direct search forms (the packer's levels);
 * the tensor cores form E (G/T) with fp32 accumulation, and each accumulator
 * column is multiplied by the matching residual column and summed (fp32 per
 * 32 columns, fp64 across them).  Arguments as awq_search_scale, with G from
 * awq_gram in place of the calibration tokens; workspace >=
 * awq_search_gram_workspace_size(N, K, n_alpha) bytes, queried on the device
 * that runs the call (it holds two 128 x 512 fp16 residual tiles per SM). */
size_t awq_search_gram_workspace_size(int64_t N, int64_t K, int n_alpha);
awq_status awq_search_scale_gram(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                 const uint16_t* G, const double* mean_abs, const double* alphas,
                                 int n_alpha, int group, float* s_out, double* mse_out,
                                 int32_t* best_idx, float* s_alpha_out, void* workspace,
                                 size_t ws_bytes, awq_stream_t stream);
/* The Gram-route search at 3 bits (levels 0..7 as awq_search_scale_int3). */
awq_status awq_search_scale_gram_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                      const uint16_t* G, const double* mean_abs,
                                      const double* alphas, int n_alpha, int group, float* s_out,
                                      double* mse_out, int32_t* best_idx, float* s_alpha_out,
                                      void* workspace, size_t ws_bytes, awq_stream_t stream);

/* ---- alpha search without any device allocation ---------------------------
 * No counterpart on the AWQ pages: an allocation-free variant of
 * awq_search_scale for callers that cannot allocate device memory (plug-ins
 * of a host program that owns the whole device memory pool; loops that must
 * avoid cudaMalloc because it can synchronise the device).  Same arguments
 * and results as awq_search_scale without the workspace: the scratch is a
 * library-owned device array of AWQ_SEARCH_NOALLOC_SCRATCH_BYTES that every
 * GPU loading the library holds until the process exits.  Problems whose
 * awq_search_workspace_size() exceeds that size are refused with
 * AWQ_ERR_WORKSPACE (bad sizes or n_alpha are AWQ_ERR_INVALID_ARG first).
 * The first call on a device looks up the array's device address (make that
 * first call before any stream capture); a call in a context other than the
 * one of that lookup (e.g. after cudaDeviceReset) looks it up again.  All
 * calls share the array: calls that overlap on the GPU race. */
#define AWQ_SEARCH_NOALLOC_SCRATCH_BYTES (16u << 20)
awq_status awq_search_scale_noalloc(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                    const uint16_t* Xcal, int64_t T, int64_t ldx,
                                    const double* mean_abs, const double* alphas, int n_alpha,
                                    int group, float* s_out, double* mse_out, int32_t* best_idx,
                                    float* s_alpha_out, awq_stream_t stream);

/* ---- step: INT4 packing --------------------------------------------------
 * Low-bit weights (third paragraph: all stored weights are low-bit; last
 * paragraph: 4 bits).  Per row n and group g of 128 input channels:
 *   w'_k  = fp32(W[n,k] * s_k)                     (s_k = 1 when s is NULL)
 *   lo,hi = min, max of w' over the group
 *   scale = fp16_rn(max(fp32(fp32(hi - lo) / 15), 2^-14))
 *   z     = clamp(rint(fp32(-lo / scale)), 0, 15)
 *   q_k   = clamp(rint(fp32(w'_k / scale)) + z, 0, 15)     (rint: ties to even)
 * and dequantisation is (q - z) * scale.
 *   W        [N, K] fp16, leading dimension ldw.
 *   s        [K] fp32 (from awq_search_scale) or NULL for plain rounding.
 *   group    must be 128.
 *   qweight  [N, K/8] uint32: element k of row n in word k/8 of that row,
 *            bits 4*(k%8) .. 4*(k%8)+3.
 *   scales   [N, K/128] fp16.     zeros [N, K/128] fp16 holding 0..15.
 * K % 128 == 0; pointers 16-byte aligned (scales/zeros: 2-byte). */
awq_status awq_pack_int4(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                         const float* s, int group, uint32_t* qweight, uint16_t* scales,
                         uint16_t* zeros, awq_stream_t stream);

/* ---- step: 3-bit packing ---------------------------------------------------
 * The pages evaluate the method at 3 and 4 bits (fourth paragraph; last
 * paragraph: 3 bits possible, with a noticeable gap).  The quantiser of
 * awq_pack_int4 with levels 0..7:
 *   scale = fp16_rn(max(fp32(fp32(hi - lo) / 7), 2^-14))
 *   z     = clamp(rint(fp32(-lo / scale)), 0, 7)
 *   q_k   = clamp(rint(fp32(w'_k / scale)) + z, 0, 7)
 *   planes   [N, 3K/32] uint32: levels 32 j .. 32 j + 31 of a row sit in
 *            words 3 j .. 3 j + 2 of that row; word 3 j + p holds bit p of
 *            level 32 j + i at bit i (exactly 3 bits per weight).
 *   scales   [N, K/128] fp16.     zeros [N, K/128] fp16 holding 0..7.
 * K % 128 == 0; W and s 16-byte aligned, planes 4-byte, scales/zeros 2-byte.
 * w3a16_gemm consumes this format. */
awq_status awq_pack_int3(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                         const float* s, int group, uint32_t* planes, uint16_t* scales,
                         uint16_t* zeros, awq_stream_t stream);

/* ---- step: 3-bit matmul ---------------------------------------------------------
 * Y = X deq(Wq)^T over the 3-bit format of awq_pack_int3, deq = (q - z) *
 * scale, fp32 accumulation, fp16 out.  For 1 <= M <= 16 tokens (decoding,
 * the memory-bound case; AWQ page sixth paragraph: fewer bytes per weight,
 * faster tokens at small batch) the planes are streamed and the products
 * summed per group; for M > 16 (AWQ page ninth paragraph: larger batches
 * are compute-bound) the tcgen05 tensor-core GEMM runs with a producer that
 * rebuilds each (q - z) exactly in fp16 and rounds (q - z) * scale once to
 * fp16.  Arguments as w4a16_gemm, with planes [N, 3K/32] uint32 in place of
 * qweight and no workspace.  X 16-byte aligned, ldx a multiple of 8; planes
 * 4-byte aligned (16-byte for M > 16). */
awq_status w3a16_gemm(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                      const uint32_t* planes, const uint16_t* scales, const uint16_t* zeros,
                      int64_t N, int group, uint16_t* Y, int64_t ldy, awq_stream_t stream);

/* ---- step: dequantise-fused matmul -----------------------------------------
 * Y = X deq(Wq)^T, deq = (q - z) * scale, fp32 accumulation, fp16 out
 * (pages: fused 4-bit kernels; on-the-fly dequantisation; memory-bound
 * decoding at small batch, more compute-bound at large batch).
 *   X        [M, K] fp16, leading dimension ldx (>= K, multiple of 8); the
 *            caller has already divided X by s (the pages' "divide its input
 *            by s", normally folded into the previous operation).
 *   qweight, scales, zeros: as written by awq_pack_int4 for an [N, K] weight.
 *   Y        [M, N] fp16, leading dimension ldy (>= N).
 * M <= 16 runs the decode kernel (packed weights streamed once, dequantised
 * in registers); M > 16 runs the tcgen05 tensor-core kernel, one 128-row x
 * 256-token output tile per CTA in turn.  When the tiles would leave the
 * grid under-filled, either every tile's K range is split over several CTAs
 * or (stream-K tail) the whole waves of tiles run as they are and the K
 * range of the remaining tiles is cut into one equal share per SM; in both
 * cases the fp32 partials go to the workspace and are added in a fixed
 * order (repeated calls give identical results).
 * workspace >= w4a16_gemm_workspace_size(M, N, K) bytes on the device that
 * runs the call (may be 0/NULL when that size is 0; 16-byte aligned).
 * K % 128 == 0, N % 8 == 0, group == 128. */
awq_status w4a16_gemm(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                      const uint32_t* qweight, const uint16_t* scales, const uint16_t* zeros,
                      int64_t N, int group, uint16_t* Y, int64_t ldy, void* workspace,
                      size_t ws_bytes, awq_stream_t stream);
size_t w4a16_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* ---- dequantise-fused matmul with the input scaling fused -----------------
 * The AWQ page's scaling trick divides each input channel by s (third
 * paragraph); the OpenAlex record's abstract names kernel fusion.  Here the
 * division is part of the matmul:
 *   Y = fp16(fp32(X) * inv_s) deq(Wq)^T,
 * each scaled activation rounded once to fp32 and once to fp16, then used
 * exactly as w4a16_gemm uses X (so the result equals w4a16_gemm on those
 * fp16 values).  For M <= 16 the scaling happens as the decode kernel stages
 * its activations; for M > 16 a pre-pass writes the scaled activations into
 * the workspace, and the tensor-core matmul, launched as its programmatic
 * dependent, starts dequantising weights while the pre-pass runs (the
 * pre-pass writes only the workspace).
 *   X      [M, K] fp16 unscaled, leading dimension ldx.
 *   inv_s  [K] fp32 device, 1/s per input channel (16-byte aligned).
 *   other arguments as w4a16_gemm; workspace >=
 *   w4a16_gemm_scaled_workspace_size(M, N, K) bytes. */
awq_status w4a16_gemm_scaled(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                             const float* inv_s, const uint32_t* qweight, const uint16_t* scales,
                             const uint16_t* zeros, int64_t N, int group, uint16_t* Y, int64_t ldy,
                             void* workspace, size_t ws_bytes, awq_stream_t stream);
size_t w4a16_gemm_scaled_workspace_size(int64_t M, int64_t N, int64_t K);

/* ---- weight packing for the decode kernel: repacked tiles ------------------
 * The OpenAlex record's abstract names weight packing for the inference
 * kernels; the AWQ page's first paragraph: decoding is memory-bound.  The
 * plain layout of awq_pack_int4 spreads the 16 rows a decode warp works on
 * over the matrix; the repack gathers each (16-row slab, group of 128) into
 * one contiguous 1088-byte tile, so the decode matmul streams contiguous
 * bytes.  Tile (j, g) of slab j (rows 16 j .. 16 j + 15) and group g sits at
 * byte (j * (K/128) + g) * 1088:
 *   bytes [0, 1024): chunk c = 32 h + L (h = 0, 1; L = 0..31) of 16 bytes is
 *     bytes 64 g + 16 (L % 4) .. +15 of row 16 j + L / 4 + 8 h of qweight
 *     (i.e. its words 16 g + 4 (L % 4) .. +3);
 *   bytes [1024, 1088): for r = 0..7, 8 bytes: the fp16 scale and zero-point
 *     of row 16 j + r, then those of row 16 j + r + 8.
 * Rows at or past N are zero.  Nothing is rounded or changed: the tiles hold
 * the same packed words, scales and zero-points.
 *   qweight, scales, zeros: as written by awq_pack_int4 for an [N, K] weight.
 *   tiles    device buffer of at least awq_repack_int4_bytes(N, K) bytes,
 *            16-byte aligned (written completely).
 * K % 128 == 0, group == 128; qweight 16-byte aligned. */
size_t awq_repack_int4_bytes(int64_t N, int64_t K);
awq_status awq_repack_int4(const uint32_t* qweight, const uint16_t* scales, const uint16_t* zeros,
                           int64_t N, int64_t K, int group, void* tiles, size_t tiles_bytes,
                           awq_stream_t stream);

/* Y = X deq(Wq)^T for 1 <= M <= 16 tokens over the repacked tiles, with the
 * arithmetic of w4a16_gemm's decode kernel (deq = (q - z) * scale, exact fp16
 * (q - z), fp32 accumulation per group, the group scale applied in fp32,
 * fp16 out) and the packed bytes streamed contiguously (AWQ page, first
 * paragraph: memory-bound decoding).  The split of K over warps depends only
 * on N and K, so results are deterministic; they may differ from
 * w4a16_gemm's in the last fp32 roundings (another split).
 *   X      [M, K] fp16, leading dimension ldx (>= K, multiple of 8).
 *   inv_s  [K] fp32 or NULL: when given, X is used as fp16(fp32(X) * inv_s)
 *          (the fused input scaling of w4a16_gemm_scaled).
 *   tiles  from awq_repack_int4 for an [N, K] weight; N % 8 == 0.
 *   Y      [M, N] fp16, leading dimension ldy (>= N).
 * M > 16 returns AWQ_ERR_SHAPE.  No workspace.  X, tiles, inv_s 16-byte
 * aligned.  Weight prefetch follows awq_set_weight_prefetch. */
awq_status w4a16_gemm_repacked(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                               const float* inv_s, const void* tiles, int64_t N, int group,
                               uint16_t* Y, int64_t ldy, awq_stream_t stream);

/* The same repack at 3 bits: tile (j, g) of awq_pack_int3's planes at byte
 * (j * (K/128) + g) * 832:
 *   bytes [0, 768): 16 rows x 48 bytes: row 16 j + r's plane words
 *     12 g .. 12 g + 11 at 48 r (rows at or past N zero);
 *   bytes [768, 832): scales and zero-points as in the 4-bit tile.
 * planes 16-byte aligned; tiles >= awq_repack_int3_bytes(N, K) bytes. */
size_t awq_repack_int3_bytes(int64_t N, int64_t K);
awq_status awq_repack_int3(const uint32_t* planes, const uint16_t* scales, const uint16_t* zeros,
                           int64_t N, int64_t K, int group, void* tiles, size_t tiles_bytes,
                           awq_stream_t stream);

/* Y = X deq(Wq)^T for 1 <= M <= 16 over the 3-bit tiles (the arithmetic of
 * w3a16_gemm's tensor-core decode: exact fp16 (q - z) pairs from the planes,
 * fp32 accumulation per group, the scale in fp32, fp16 out; AWQ page sixth
 * paragraph: fewer bytes per weight, faster small-batch tokens).  Arguments
 * as w4a16_gemm_repacked without inv_s.  M > 16 returns AWQ_ERR_SHAPE. */
awq_status w3a16_gemm_repacked(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                               const void* tiles, int64_t N, int group, uint16_t* Y, int64_t ldy,
                               awq_stream_t stream);

/* Overlap of back-to-back matmuls.  Every decode launch (M <= 16) lets the
 * next kernel in the stream start beside it (programmatic dependent launch),
 * and every matmul launch (decode and tensor-core) may start beside the
 * previous kernel; each reads X / writes Y only after the previous kernel in
 * the stream has completed.  With enable = 1 a matmul also starts fetching
 * (decode) or dequantising (M > 16) its packed weights (qweight or planes,
 * scales, zeros; the repacked tiles) before that point, so consecutive
 * matmuls keep HBM busy across kernel boundaries, as in a decode step where
 * the weights are constant.  Enable it only if no kernel that writes a
 * matmul's packed weights (awq_pack_int4 or any other) is the kernel
 * immediately before that matmul call in its stream; otherwise the matmul
 * may read stale weights.
 * Process-wide setting, default 0.  Returns AWQ_ERR_INVALID_ARG unless
 * enable is 0 or 1.  (Host-side setting; the pages describe no counterpart
 * beyond memory-bound decoding with fused 4-bit kernels.) */
awq_status awq_set_weight_prefetch(int enable);

/* ---- status and diagnostics ---------------------------------------------- */

/* Synchronise `stream`, then return (and clear) the device-side status word
 * of the current device: AWQ_OK, AWQ_ERR_NONFINITE, AWQ_ERR_OVERFLOW or
 * AWQ_ERR_TIMEOUT (the most severe seen since the last call, in the order
 * timeout, overflow, non-finite), or AWQ_ERR_CUDA if the synchronisation
 * itself failed. */
awq_status awq_sync_status(awq_stream_t stream);

/* Diagnostic of the failure path (no counterpart on the AWQ pages): every
 * device-side wait in the library's kernels is bounded, and a wait that runs
 * out records AWQ_ERR_TIMEOUT in the status word and lets the kernel return,
 * so the context stays usable.  This call launches one small kernel whose
 * bounded wait, limited to limit_us microseconds (1 .. 1e6), is on a barrier
 * that nothing arrives on; awq_sync_status() then returns AWQ_ERR_TIMEOUT
 * (and clears it).  Nothing faults, traps or hangs. */
awq_status awq_selftest_wait_timeout(int64_t limit_us, awq_stream_t stream);

/* Static text for the last error returned by a call on this host thread. */
const char* awq_last_error_string(void);

/* Library version as major*10000 + minor*100 + patch. */
int awq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* AWQ_B300_H */
