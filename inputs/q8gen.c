/*
 * Seeded synthetic input generator for the Q8_0 x Q8_0 matmul workloads.
 *
 * This module is shared by the test oracle and by the CUDA path's tests and
 * benchmark.  It holds none of the method's arithmetic: it only draws numbers.
 * Every value is a pure function of (seed, stream, element index), so any
 * slice can be produced independently and in parallel.  The integer draws,
 * weights and routing are identical on every platform; the N(0,1) values go
 * through the C library's log1p, cos and sqrt and may differ in the last bit
 * between C libraries (both sides of a comparison always use the same arrays).
 *
 * Random source: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), used in its counter form:
 * output i of a stream is the SplitMix64 finaliser applied to
 * key + (i + 1) * golden_gamma.
 *
 * Distributions (the workloads of the "Q8_0 matmul" trace, ds4 GPU code
 * walkthrough, trace 3, and the MoE section of the model-architecture page):
 *   - weights: Q8_0 rows of 34-byte blocks (fp16 d little-endian, then 32 int8 q);
 *     q uniform over the 255 values -127..127 (multiply-shift range reduction of
 *     a 32-bit draw, Lemire 2019; bias below 2^-24), d uniform in [1e-3, 1e-2]
 *     drawn in double and rounded to the nearest binary16 value (ties to even).
 *   - activations: N(0,1) by the Box-Muller transform on two uniform draws,
 *     rounded to float; optionally each element independently scaled by a
 *     factor with a given probability (outliers).
 *   - routing: k distinct experts per token, uniform (partial Fisher-Yates) or
 *     Zipf(s) over ranks 1..n_expert (rank r -> expert r-1) by sequential
 *     weighted draws without replacement.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of a stream: the seed and the stream id mixed once. */
static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return sm64_mix(seed ^ sm64_mix(stream + GOLDEN_GAMMA));
}

/* Draw i (0-based) of the stream with the given key. */
static inline uint64_t draw(uint64_t key, uint64_t i) {
    return sm64_mix(key + (i + 1) * GOLDEN_GAMMA);
}

/* Uniform double in [0, 1) from the top 53 bits. */
static inline double unit(uint64_t r) {
    return (double)(r >> 11) * (1.0 / 9007199254740992.0);
}

/* Nearest binary16 (ties to even) of a positive double in the normal range
 * [2^-14, 65504]; used only to place the weight scales on the fp16 grid. */
static uint16_t to_half_grid(double v) {
    int e;
    double m = frexp(v, &e);            /* v = m * 2^e, m in [0.5, 1) */
    int E = e - 1;                      /* v = (2m) * 2^E, 2m in [1, 2) */
    double f = nearbyint(m * 2048.0 - 1024.0); /* 10-bit fraction, RN-even */
    if (f >= 1024.0) { f = 0.0; E += 1; }
    return (uint16_t)(((unsigned)(E + 15) << 10) | (unsigned)f);
}

int q8g_version(void) { return 1; }

/* Raw Q8_0 weight rows: rows x (in_dim/32) blocks of 34 bytes. */
int q8g_weights(uint8_t *W, uint64_t rows, uint64_t in_dim, uint64_t seed,
                uint64_t stream, double d_lo, double d_hi) {
    if (!W || in_dim % 32) return -1;
    const uint64_t nb = in_dim / 32;
    const uint64_t nblk = rows * nb;
    const uint64_t kd = stream_key(seed, 2 * stream);      /* scales */
    const uint64_t kq = stream_key(seed, 2 * stream + 1);  /* quants */
    #pragma omp parallel for schedule(static)
    for (int64_t blk = 0; blk < (int64_t)nblk; ++blk) {
        uint8_t *p = W + (uint64_t)blk * 34;
        double v = d_lo + (d_hi - d_lo) * unit(draw(kd, (uint64_t)blk));
        uint16_t h = to_half_grid(v);
        p[0] = (uint8_t)(h & 0xff);
        p[1] = (uint8_t)(h >> 8);
        for (int i = 0; i < 32; i += 2) {
            uint64_t r = draw(kq, (uint64_t)blk * 16 + (uint64_t)(i / 2));
            uint32_t lo = (uint32_t)r, hi = (uint32_t)(r >> 32);
            int a = (int)(((uint64_t)lo * 255u) >> 32) - 127;
            int b = (int)(((uint64_t)hi * 255u) >> 32) - 127;
            p[2 + i] = (uint8_t)(int8_t)a;
            p[3 + i] = (uint8_t)(int8_t)b;
        }
    }
    return 0;
}

/* Raw K-quant weight rows: rows x (in_dim/256) blocks of 84 (fmt 2, Q2_K) or
 * 144 (fmt 4, Q4_K) bytes.  d and dmin are drawn uniformly from [d_lo, d_hi]
 * and [m_lo, m_hi] (both within the binary16 normal range) and placed on the
 * binary16 grid at the block's d and dmin bytes; every other byte (scales,
 * mins, quants) is uniform. */
int q8g_kq_weights(uint8_t *W, uint64_t rows, uint64_t in_dim, int fmt, uint64_t seed, uint64_t stream,
                   double d_lo, double d_hi, double m_lo, double m_hi) {
    if (!W || in_dim % 256 || (fmt != 2 && fmt != 4) || d_lo < 0x1p-14 || m_lo < 0x1p-14) return -1;
    const uint64_t bb = fmt == 2 ? 84 : 144;
    const uint64_t d_off = fmt == 2 ? 80 : 0;
    const uint64_t nblk = rows * (in_dim / 256);
    const uint64_t kd = stream_key(seed, 100 + 2 * stream);   /* d, dmin */
    const uint64_t kb = stream_key(seed, 101 + 2 * stream);   /* the other bytes */
    #pragma omp parallel for schedule(static)
    for (int64_t blk = 0; blk < (int64_t)nblk; ++blk) {
        uint8_t *p = W + (uint64_t)blk * bb;
        for (uint64_t i = 0; i < bb; i += 8) {
            uint64_t r = draw(kb, (uint64_t)blk * 24 + i / 8);
            for (uint64_t j = 0; j < 8 && i + j < bb; ++j) p[i + j] = (uint8_t)(r >> (8 * j));
        }
        uint16_t h = to_half_grid(d_lo + (d_hi - d_lo) * unit(draw(kd, 2 * (uint64_t)blk)));
        uint16_t hm = to_half_grid(m_lo + (m_hi - m_lo) * unit(draw(kd, 2 * (uint64_t)blk + 1)));
        p[d_off] = (uint8_t)(h & 0xff);
        p[d_off + 1] = (uint8_t)(h >> 8);
        p[d_off + 2] = (uint8_t)(hm & 0xff);
        p[d_off + 3] = (uint8_t)(hm >> 8);
    }
    return 0;
}

/* N(0,1) activations; with probability p_out an element is multiplied by
 * out_scale (p_out = 0 disables). */
int q8g_normal(float *x, uint64_t n, uint64_t seed, uint64_t stream,
               double p_out, double out_scale) {
    if (!x && n) return -1;
    const uint64_t ku = stream_key(seed, 2 * stream);
    const uint64_t ko = stream_key(seed, 2 * stream + 1);
    const double two_pi = 6.283185307179586476925286766559;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < (int64_t)n; ++i) {
        double u1 = unit(draw(ku, 2 * (uint64_t)i));
        double u2 = unit(draw(ku, 2 * (uint64_t)i + 1));
        double z = sqrt(-2.0 * log1p(-u1)) * cos(two_pi * u2);
        if (p_out > 0.0 && unit(draw(ko, (uint64_t)i)) < p_out) z *= out_scale;
        x[i] = (float)z;
    }
    return 0;
}

/* k distinct experts per token, uniform over n_expert (partial Fisher-Yates). */
int q8g_route_uniform(int32_t *ids, uint64_t n_tok, uint32_t k,
                      uint32_t n_expert, uint64_t seed, uint64_t stream) {
    if (!ids || k == 0 || k > n_expert) return -1;
    const uint64_t key = stream_key(seed, stream);
    int failed = 0;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < (int64_t)n_tok; ++t) {
        int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * n_expert);
        if (!perm) {
            #pragma omp atomic write
            failed = 1;
            continue;
        }
        for (uint32_t e = 0; e < n_expert; ++e) perm[e] = (int32_t)e;
        for (uint32_t j = 0; j < k; ++j) {
            uint64_t r = draw(key, (uint64_t)t * k + j);
            uint32_t span = n_expert - j;
            uint32_t pick = j + (uint32_t)(((r >> 32) * (uint64_t)span) >> 32);
            int32_t tmp = perm[j]; perm[j] = perm[pick]; perm[pick] = tmp;
            ids[(uint64_t)t * k + j] = perm[j];
        }
        free(perm);
    }
    return failed ? -1 : 0;
}

/* k distinct experts per token, Zipf(s): P(rank r) proportional to r^-s,
 * rank r -> expert r-1; sequential weighted draws without replacement. */
int q8g_route_zipf(int32_t *ids, uint64_t n_tok, uint32_t k, uint32_t n_expert,
                   double s, uint64_t seed, uint64_t stream) {
    if (!ids || k == 0 || k > n_expert) return -1;
    const uint64_t key = stream_key(seed, stream);
    double *w0 = (double *)malloc(sizeof(double) * n_expert);
    if (!w0) return -1;
    for (uint32_t r = 0; r < n_expert; ++r) w0[r] = pow((double)(r + 1), -s);
    int failed = 0;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < (int64_t)n_tok; ++t) {
        double *w = (double *)malloc(sizeof(double) * n_expert);
        if (!w) {
            #pragma omp atomic write
            failed = 1;
            continue;
        }
        memcpy(w, w0, sizeof(double) * n_expert);
        for (uint32_t j = 0; j < k; ++j) {
            double total = 0.0;
            for (uint32_t r = 0; r < n_expert; ++r) total += w[r];
            double target = unit(draw(key, (uint64_t)t * k + j)) * total;
            uint32_t pick = n_expert;
            double acc = 0.0;
            for (uint32_t r = 0; r < n_expert; ++r) {
                if (w[r] == 0.0) continue;
                acc += w[r];
                pick = r;
                if (target < acc) break;
            }
            ids[(uint64_t)t * k + j] = (int32_t)pick;
            w[pick] = 0.0;
        }
        free(w);
    }
    free(w0);
    return failed ? -1 : 0;
}
