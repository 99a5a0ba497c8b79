/*
 * Seeded synthetic inputs for the direct-access decode kernels and their oracle.
 *
 * This file holds no arithmetic of the method itself: it only turns (seed, stream,
 * element index) into bf16 bit patterns. Both the CUDA path and the CPU oracle read
 * the same bytes, so neither depends on the other.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014) used as a counter-based hash: value i of a stream is the
 * SplitMix64 output mix applied to key + (i + 1) * golden_gamma. Normals come from the
 * Box-Muller transform (Box and Muller, 1958) in double precision, one 64-bit draw per
 * pair of normals. Values are rounded to bf16 with round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GOLDEN_GAMMA) ^ (stream * 0xD1B54A32D192ED03ULL + 1ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1ULL) * GOLDEN_GAMMA);
}

/* float -> bf16 bits, round to nearest even; NaN stays NaN. */
static inline uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    uint64_t r = draw(key, i >> 1);
    /* two open-interval uniforms from the two 32-bit halves */
    double u1 = ((double)(r >> 32) + 0.5) * (1.0 / 4294967296.0);
    double u2 = ((double)(r & 0xFFFFFFFFULL) + 0.5) * (1.0 / 4294967296.0);
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586476925286766559 * u2;
    return (i & 1ULL) ? rad * sin(ang) : rad * cos(ang);
}

/* out[j] = bf16(mean + std * N(0,1)_{offset + j}) for j < n */
void synth_normal_bf16(uint64_t seed, uint64_t stream, double mean, double std,
                       uint64_t offset, uint64_t n, uint16_t *out) {
    uint64_t key = stream_key(seed, stream);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < nn; ++j) {
        double v = mean + std * normal_at(key, offset + (uint64_t)j);
        out[j] = to_bf16((float)v);
    }
}

/* out[j] = bf16 of an integer drawn uniformly from [lo, hi] (exact in bf16 for |v| <= 256) */
void synth_int_bf16(uint64_t seed, uint64_t stream, int lo, int hi,
                    uint64_t offset, uint64_t n, uint16_t *out) {
    uint64_t key = stream_key(seed, stream);
    uint64_t span = (uint64_t)(hi - lo + 1);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < nn; ++j) {
        uint64_t r = draw(key, offset + (uint64_t)j);
        int v = lo + (int)((r >> 11) % span);
        out[j] = to_bf16((float)v);
    }
}

/* out[j] = uniform double in [0, 1) for j < n (used for shuffles and small test choices) */
void synth_uniform_f64(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, double *out) {
    uint64_t key = stream_key(seed, stream);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < nn; ++j) {
        uint64_t r = draw(key, offset + (uint64_t)j);
        out[j] = (double)(r >> 11) * (1.0 / 9007199254740992.0);
    }
}

/* worker threads this library will use (OpenMP), reported with CPU timings */
int synth_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
