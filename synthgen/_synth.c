/* Counter-based random draws for the synthetic workloads: SplitMix64 words
 * and Box-Muller normals.  Holds no arithmetic of the quantisation method.
 * Output depends only on (seed, index), never on the thread count. */
#include <math.h>
#include <stdint.h>

static inline uint64_t sm64_word(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

void sg_splitmix64(uint64_t seed, uint64_t offset, int64_t n, uint64_t* out) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = sm64_word(seed, offset + (uint64_t)i);
}

/* Normals offset .. offset+n-1 of stream seed, each multiplied by `scale`.
 * Normal 2j uses r*cos, normal 2j+1 uses r*sin, from words 2j and 2j+1. */
void sg_normals(uint64_t seed, int64_t offset, int64_t n, double scale, double* out) {
    const double two_pi = 6.283185307179586476925286766559;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t idx = (uint64_t)(offset + i);
        uint64_t j = idx >> 1;
        uint64_t w0 = sm64_word(seed, 2 * j), w1 = sm64_word(seed, 2 * j + 1);
        double u1 = (double)((w0 >> 11) + 1) * 0x1p-53;
        double u2 = (double)(w1 >> 11) * 0x1p-53;
        double r = sqrt(-2.0 * log(u1));
        double th = two_pi * u2;
        double v = (idx & 1) ? r * sin(th) : r * cos(th);
        out[i] = scale * v;
    }
}
