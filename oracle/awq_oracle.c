/*
 * AWQ hot path: plain, slow CPU oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the bench's CPU-baseline / reference
 * legs may load this file's library.  It shares no code, header or constant
 * table with the CUDA library and never calls it.
 *
 * Sources (the AWQ pages):
 *   - "AWQ: Activation-aware Weight Quantization for On-Device LLM Compression
 *     and Acceleration" (fdeinterviews.com/papers/awq), third paragraph: a
 *     weight channel is scaled up by s > 1 and its input down by s; s is a
 *     power alpha of the channel's mean absolute activation; alpha is picked
 *     by trying a small grid on a few calibration samples; all stored
 *     weights are low-bit.  Seventh paragraph: the method gathers activation
 *     statistics and fits nothing.
 *     Fourth paragraph: the method was evaluated at 3 and 4 bits; last
 *     paragraph: 4 bits is the default, 3 bits possible with a noticeable
 *     gap.
 *   - Group size 128, asymmetric levels 0..15 (0..7 at 3 bits) with an fp16
 *     scale and fp16 zero-point per group, 8 nibbles per uint32 (3 bit
 *     planes per 32 levels at 3 bits), mean |x| as the average magnitude,
 *     output MSE as the search objective and the 20-point alpha grid are
 *     not on the pages; they are the stated workload definition.
 *
 * Every value the method rounds is rounded at exactly one stated point:
 * "fp32(expr)" means expr is evaluated exactly or in fp64 and then rounded
 * once to fp32 (ties to even).  For a single +, -, *, / of fp32/fp16
 * operands this equals the IEEE fp32 operation, because 53 >= 2*24 + 2.
 * Built with -ffp-contract=off and without fast-math, so no FMA contraction
 * or reassociation happens.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GROUP 128

enum { OR_OK = 0, OR_ERR_ARG = 1, OR_ERR_NONFINITE = 8 };

/* ---- IEEE 754 binary16, written from the format's definition ---------- */

/* Exact value of an fp16 bit pattern. */
double awqo_h2d(uint16_t h) {
    int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp((double)(1024 + f), e - 25);          /* (1 + f/1024) 2^(e-15) */
    return sign ? -v : v;
}

/* Nearest fp16 to x, ties to even; overflow gives +-Inf. */
uint16_t awqo_d2h_rn(double x) {
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a < 0x1p-14) {                                   /* subnormal range */
        double r = rint(ldexp(a, 24));                   /* units of 2^-24, exact scaling */
        return sign | (uint16_t)r;                       /* r == 1024 is the least normal */
    }
    int p;
    frexp(a, &p);                                        /* a = m 2^p, m in [0.5, 1) */
    int E = p - 1;                                       /* a in [2^E, 2^(E+1)) */
    double r = rint(ldexp(a, 10 - E));                   /* in [1024, 2048] */
    if (r == 2048.0) { r = 1024.0; E += 1; }
    if (E > 15) return sign | 0x7C00;
    return sign | (uint16_t)((E + 15) << 10) | (uint16_t)(r - 1024.0);
}

/* fp16 -> integer multiple of 2^-24 (exact for finite values); -1 for Inf/NaN. */
static int64_t h_abs_q24(uint16_t h) {
    int e = (h >> 10) & 31, f = h & 1023;
    if (e == 31) return -1;
    if (e == 0) return f;
    return (int64_t)(1024 + f) << (e - 1);
}

/* ---- step a1: per-input-channel activation statistics ------------------ */

/* abs_sum[k] = sum_t |X[t,k]| * 2^24, an exact integer (every finite fp16 is
 * a multiple of 2^-24 below 2^16, so the sum is exact for T < 2^23).
 * accumulate = 0 overwrites, 1 adds to abs_sum. */
int awqo_act_stats(const uint16_t* X, int64_t T, int64_t K, int64_t ldx,
                   int accumulate, int64_t* abs_sum) {
    if (T < 0 || K < 0 || ldx < K) return OR_ERR_ARG;
    int bad = 0;
    for (int64_t k = 0; k < K; ++k) {
        int64_t acc = accumulate ? abs_sum[k] : 0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t v = h_abs_q24(X[t * ldx + k]);
            if (v < 0) bad = 1; else acc += v;
        }
        abs_sum[k] = acc;
    }
    return bad ? OR_ERR_NONFINITE : OR_OK;
}

/* m[k] = abs_sum[k] / 2^24 / n_tokens, both divisions in fp64. */
void awqo_act_mean(const int64_t* abs_sum, int64_t n_tokens, int64_t K, double* m) {
    for (int64_t k = 0; k < K; ++k)
        m[k] = ((double)abs_sum[k] / 16777216.0) / (double)n_tokens;
}

/* ---- step a2: candidate scales ----------------------------------------- */

/* s_k = fp32( r_k / sqrt(max_j r_j * min_j r_j) ),  r_k = pow(max(m_k, 1e-4), alpha).
 * The normaliser only keeps s near 1: dividing s by any constant leaves the
 * quantised layer's output unchanged. */
void awqo_candidate_scales(const double* m, int64_t K, double alpha, float* s) {
    double rmax = -INFINITY, rmin = INFINITY;
    for (int64_t k = 0; k < K; ++k) {
        double r = pow(fmax(m[k], 1e-4), alpha);
        if (r > rmax) rmax = r;
        if (r < rmin) rmin = r;
    }
    double norm = sqrt(rmax * rmin);
    for (int64_t k = 0; k < K; ++k) {
        double r = pow(fmax(m[k], 1e-4), alpha);
        s[k] = (float)(r / norm);
    }
}

/* ---- steps a3/a5: quantise one row-group of 128 weights --------------- */

/* Asymmetric round-to-nearest of w' = W*s over one group, with levels
 * 0..qmax (qmax = 2^bits - 1: 15 at 4 bits, 7 at 3 bits):
 *   1. w'_k   = fp32(W_k * s_k)                   (s_k = 1 when s is NULL)
 *   2. lo, hi = min, max of w'
 *   3. d      = fp32(fp32(hi - lo) / qmax)
 *   4. scale  = fp16_rn(max(d, 2^-14))            (stored)
 *   5. z      = clamp(rint(fp32(-lo / scale)), 0, qmax)   (stored as fp16)
 *   6. q_k    = clamp(rint(fp32(w'_k / scale)) + z, 0, qmax)
 * rint is round-half-to-even.  Returns OR_ERR_NONFINITE if an input is not
 * finite or the scale overflows fp16. */
static int quant_group(const uint16_t* w, const float* s, int qmax, uint8_t* q,
                       uint16_t* scale_out, uint16_t* zero_out) {
    const float fq = (float)qmax;
    float wp[GROUP];
    for (int k = 0; k < GROUP; ++k) {
        double wk = awqo_h2d(w[k]);
        if (!isfinite(wk)) return OR_ERR_NONFINITE;
        double sk = s ? (double)s[k] : 1.0;
        wp[k] = (float)(wk * sk);                    /* exact product, one rounding */
        if (!isfinite(wp[k])) return OR_ERR_NONFINITE;
    }
    float lo = wp[0], hi = wp[0];
    for (int k = 1; k < GROUP; ++k) {
        if (wp[k] < lo) lo = wp[k];
        if (wp[k] > hi) hi = wp[k];
    }
    float range = (float)((double)hi - (double)lo);
    float d = (float)((double)range / (double)qmax);
    if (d < 0x1p-14f) d = 0x1p-14f;
    uint16_t sh = awqo_d2h_rn((double)d);
    if ((sh & 0x7C00) == 0x7C00) return OR_ERR_NONFINITE;
    double scale = awqo_h2d(sh);
    /* the zero-point is an integer level 0..qmax; the clamp maps -0 (from
     * rint of a negative quotient above -0.5) to the integer 0, i.e. +0.0 */
    float zf = rintf((float)(-(double)lo / scale));
    if (!(zf > 0.0f)) zf = 0.0f;
    if (zf > fq) zf = fq;
    for (int k = 0; k < GROUP; ++k) {
        float t = (float)((double)wp[k] / scale);
        float v = rintf(t) + zf;                     /* exact: |rint(t)| < 2^24 or clamped */
        if (v < 0.0f) v = 0.0f;
        if (v > fq) v = fq;
        q[k] = (uint8_t)v;
    }
    *scale_out = sh;
    *zero_out = awqo_d2h_rn((double)zf);
    return OR_OK;
}

/* Quantise W [N,K] (row stride ldw) with per-input-channel scales s [K]
 * (NULL: plain round-to-nearest) to `bits` bits (3 or 4).  q: [N,K] one
 * level per byte; scales, zeros: [N, K/128] fp16. */
int awqo_quantize_bits(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                       const float* s, int bits, uint8_t* q, uint16_t* scales,
                       uint16_t* zeros) {
    if (N < 0 || K < 0 || K % GROUP || ldw < K || (bits != 3 && bits != 4)) return OR_ERR_ARG;
    const int qmax = (1 << bits) - 1;
    int64_t G = K / GROUP;
    int bad = 0;
    /* rows are independent; the threads only split the row range */
    #pragma omp parallel for schedule(static) reduction(|:bad)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g) {
            int r = quant_group(W + n * ldw + g * GROUP, s ? s + g * GROUP : NULL, qmax,
                                q + n * K + g * GROUP, scales + n * G + g, zeros + n * G + g);
            if (r) bad |= r;
        }
    return bad;
}

/* The 4-bit quantiser of steps a3/a5. */
int awqo_quantize(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                  const float* s, uint8_t* q, uint16_t* scales, uint16_t* zeros) {
    return awqo_quantize_bits(W, N, K, ldw, s, 4, q, scales, zeros);
}

/* ---- packing: 8 nibbles per uint32 --------------------------------------- */

/* Element k of row n sits in word k/8 of that row, bits 4*(k%8) .. 4*(k%8)+3. */
void awqo_pack_nibbles(const uint8_t* q, int64_t N, int64_t K, uint32_t* words) {
    int64_t W8 = K / 8;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < W8; ++j) {
            uint32_t w = 0;
            for (int e = 0; e < 8; ++e) w |= (uint32_t)(q[n * K + 8 * j + e] & 15) << (4 * e);
            words[n * W8 + j] = w;
        }
}

void awqo_unpack_nibbles(const uint32_t* words, int64_t N, int64_t K, uint8_t* q) {
    int64_t W8 = K / 8;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            q[n * K + k] = (uint8_t)((words[n * W8 + k / 8] >> (4 * (k % 8))) & 15);
}

/* ---- 3-bit packing: three bit planes per 32 levels ----------------------
 * Levels k = 32 j .. 32 j + 31 of row n occupy words 3 j, 3 j + 1, 3 j + 2 of
 * that row; word 3 j + p holds bit p of level 32 j + i at bit i.  Exactly 3
 * bits per weight, and a group of 128 levels is 12 whole words. */
void awqo_pack_planes3(const uint8_t* q, int64_t N, int64_t K, uint32_t* words) {
    int64_t B = K / 32;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < B; ++j)
            for (int p = 0; p < 3; ++p) {
                uint32_t w = 0;
                for (int i = 0; i < 32; ++i)
                    w |= (uint32_t)((q[n * K + 32 * j + i] >> p) & 1) << i;
                words[(n * B + j) * 3 + p] = w;
            }
}

void awqo_unpack_planes3(const uint32_t* words, int64_t N, int64_t K, uint8_t* q) {
    int64_t B = K / 32;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const uint32_t* w = words + (n * B + k / 32) * 3;
            int i = (int)(k % 32);
            q[n * K + k] = (uint8_t)(((w[0] >> i) & 1) | (((w[1] >> i) & 1) << 1) |
                                     (((w[2] >> i) & 1) << 2));
        }
}

/* Dequantised weights in fp64: deq[n,k] = (q - z) * scale. */
void awqo_dequant(const uint8_t* q, const uint16_t* scales, const uint16_t* zeros,
                  int64_t N, int64_t K, double* deq) {
    int64_t G = K / GROUP;
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            double sc = awqo_h2d(scales[n * G + k / GROUP]);
            double z = awqo_h2d(zeros[n * G + k / GROUP]);
            deq[n * K + k] = ((double)q[n * K + k] - z) * sc;
        }
}

/* Search residual E[n,k] = (q - z) * scale / s_k - W[n,k], fp64, for one
 * candidate s (NULL: s = 1).  ||X E^T||_F^2 / (T N) is then the output MSE of
 * Q(W diag(s)) diag(s)^-1 against W on the calibration activations X. */
void awqo_search_residual(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                          const float* s, const uint8_t* q, const uint16_t* scales,
                          const uint16_t* zeros, double* E) {
    int64_t G = K / GROUP;
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            double sc = awqo_h2d(scales[n * G + k / GROUP]);
            double z = awqo_h2d(zeros[n * G + k / GROUP]);
            double sk = s ? (double)s[k] : 1.0;
            E[n * K + k] = ((double)q[n * K + k] - z) * sc / sk - awqo_h2d(W[n * ldw + k]);
        }
}

/* Exact fp16 -> fp64 widening of a whole array (for the matmul steps). */
void awqo_h2d_array(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = awqo_h2d(h[i]);
}

/* Y[m,n] = sum_k X[m,k] * deq(n,k) for a list of (m, n) pairs, fp64,
 * straight from the packed words (sampled parity at full size). */
void awqo_w4a16_pairs(const uint16_t* X, int64_t ldx, int64_t K,
                      const uint32_t* qweight, const uint16_t* scales,
                      const uint16_t* zeros, int64_t n_pairs,
                      const int64_t* ms, const int64_t* ns, double* Y) {
    int64_t G = K / GROUP, W8 = K / 8;
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < n_pairs; ++i) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            uint32_t q = (qweight[n * W8 + k / 8] >> (4 * (k % 8))) & 15;
            double sc = awqo_h2d(scales[n * G + k / GROUP]);
            double z = awqo_h2d(zeros[n * G + k / GROUP]);
            acc += awqo_h2d(X[m * ldx + k]) * (((double)q - z) * sc);
        }
        Y[i] = acc;
    }
}

/* Nearest-fp16 rounding of a whole fp64 array (bits out). */
void awqo_d2h_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = awqo_d2h_rn(x[i]);
}

/* Input scaling of the matmul: Xs[m,k] = fp16_rn(fp32(X[m,k] * inv_s[k])),
 * the product exact in fp64 and rounded once to fp32, then once to fp16. */
void awqo_scale_activations(const uint16_t* X, int64_t M, int64_t K, const float* inv_s,
                            uint16_t* Xs) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float v = (float)(awqo_h2d(X[m * K + k]) * (double)inv_s[k]);
            Xs[m * K + k] = awqo_d2h_rn((double)v);
        }
}
