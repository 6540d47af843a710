/*
 * synth.c - seeded synthetic inputs for the routed-MoE workloads.
 *
 * This module produces INPUTS only: random bytes, random floats and random
 * permutations.  It contains none of the method's arithmetic (no block
 * decoding, no routing, no expert math); the oracle and the CUDA library each
 * do that on their own.  Both sides receive identical bytes from here.
 *
 * Generator: counter-based SplitMix64.  The output function is the published
 * SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014, with the mixing constants Vigna uses in
 * splitmix64.c).  Draw i of the stream with state `key` is
 * mix64(key + (i + 1) * 0x9E3779B97F4A7C15), i.e. exactly the i-th output of
 * a SplitMix64 generator seeded with `key`, but addressable at random.
 *
 * Cross-machine reproducibility: everything here uses IEEE basic operations
 * (+, -, *, /, sqrt) plus exact bit manipulation (frexp, ldexp, floor), and
 * the file is compiled with -ffp-contract=off, so x86-64 and aarch64 produce
 * the same bits.  The logarithm and sine/cosine needed for normal deviates
 * are therefore computed by short series below instead of libm.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

enum { TAG_GRID = 1, TAG_ROUTER = 2, TAG_QBLK = 3, TAG_X = 4, TAG_ZIPF = 5, TAG_RESID = 6 };

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}
uint64_t synth_mix64(uint64_t z) { return mix64(z); }

/* Stream key for (seed, purpose tag, a, b); a and b are e.g. layer and expert. */
uint64_t synth_key(uint64_t seed, uint32_t tag, uint64_t a, uint64_t b) {
    uint64_t k = mix64(seed + SYNTH_GOLDEN * ((uint64_t)tag + 1));
    k = mix64(k + SYNTH_GOLDEN * (a + 1));
    return mix64(k + SYNTH_GOLDEN * (b + 1));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + SYNTH_GOLDEN * (i + 1)); }
uint64_t synth_draw(uint64_t key, uint64_t i) { return draw(key, i); }

static inline double unit_co(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }        /* [0,1) */
static inline double unit_oc(uint64_t r) { return (double)((r >> 11) + 1) * 0x1.0p-53; }  /* (0,1] */
/* integer in [0, n) by multiply-shift on the high 32 bits (n < 2^32) */
static inline uint32_t below(uint64_t r, uint32_t n) { return (uint32_t)(((r >> 32) * (uint64_t)n) >> 32); }

/* Natural logarithm for finite u > 0: u = m 2^e with m in [1/sqrt2, sqrt2),
 * ln m = 2 atanh(s), s = (m-1)/(m+1), |s| < 0.172, series to s^41. */
double synth_ln(double u) {
    int e;
    double m = frexp(u, &e);
    if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
    double s = (m - 1.0) / (m + 1.0);
    double s2 = s * s, term = s, sum = 0.0;
    for (int k = 1; k <= 41; k += 2) { sum += term / (double)k; term *= s2; }
    return 2.0 * sum + (double)e * 0.69314718055994530942;
}

/* sin and cos of 2*pi*v for v in [0,1): quadrant split, then Taylor series on [0, pi/2). */
void synth_sincos2pi(double v, double *s_out, double *c_out) {
    double t = v * 4.0;
    int q = (int)t;
    double th = (t - (double)q) * 1.57079632679489661923;
    double th2 = th * th, ts = th, tc = 1.0, sn = 0.0, cs = 0.0;
    for (int k = 0; k < 13; k++) {
        sn += ts; cs += tc;
        ts *= -th2 / (double)((2 * k + 2) * (2 * k + 3));
        tc *= -th2 / (double)((2 * k + 1) * (2 * k + 2));
    }
    switch (q & 3) {
        case 0: *s_out = sn;  *c_out = cs;  break;
        case 1: *s_out = cs;  *c_out = -sn; break;
        case 2: *s_out = -sn; *c_out = -cs; break;
        default: *s_out = -cs; *c_out = sn; break;
    }
}

/* IEEE binary16 bits of v, round-to-nearest-even (finite inputs; overflow -> inf). */
uint16_t synth_f16_bits(double v) {
    uint64_t b;
    memcpy(&b, &v, 8);
    uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);
    int E = e - 1; /* a = 1.f * 2^E */
    if (E > 15) return (uint16_t)(sign | 0x7C00u);
    double scaled = (E >= -14) ? ldexp(a, 10 - E) : ldexp(a, 24);
    double fl = floor(scaled), rem = scaled - fl;
    uint32_t q = (uint32_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (q & 1u))) q++;
    if (E < -14) return (uint16_t)(sign | q); /* subnormal; q == 1024 is the smallest normal */
    if (q == 2048u) { q = 1024u; E++; if (E > 15) return (uint16_t)(sign | 0x7C00u); }
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024u));
}

/* 256 x 8 codebook grid, entries i.i.d. uniform over {8, 25, 43}. */
void synth_grid(uint64_t seed, int8_t *out) {
    static const int8_t vals[3] = {8, 25, 43};
    uint64_t key = synth_key(seed, TAG_GRID, 0, 0);
    for (int i = 0; i < 256 * 8; i++) out[i] = vals[below(draw(key, (uint64_t)i), 3)];
}

/* nblocks 66-byte blocks of one matrix: 2 bytes of fp16 scale d ~ U[1e-3, 4e-3)
 * (little-endian), then 64 uniformly random bytes. */
void synth_matrix_blocks(uint64_t seed, int32_t layer, int32_t expert, int32_t matrix,
                         int64_t nblocks, uint8_t *out) {
    uint64_t key = synth_key(seed, TAG_QBLK, (uint64_t)layer, (uint64_t)expert * 4u + (uint64_t)matrix);
    for (int64_t j = 0; j < nblocks; j++) {
        uint8_t *blk = out + 66 * j;
        uint64_t base = 9u * (uint64_t)j;
        uint16_t d = synth_f16_bits(1e-3 + 3e-3 * unit_co(draw(key, base)));
        blk[0] = (uint8_t)(d & 0xFF);
        blk[1] = (uint8_t)(d >> 8);
        for (int w = 0; w < 8; w++) {
            uint64_t r = draw(key, base + 1 + (uint64_t)w);
            uint8_t le[8];
            for (int by = 0; by < 8; by++) le[by] = (uint8_t)(r >> (8 * by)); /* little-endian bytes */
            memcpy(blk + 2 + 8 * w, le, 8);
        }
    }
}

/* n_experts consecutive expert records [gate I x H | up I x H | down H x I] of one layer,
 * experts e0 .. e0 + n_experts - 1, written back to back (record = 3 * H*I/256 * 66 bytes). */
void synth_expert_records(uint64_t seed, int32_t layer, int32_t e0, int32_t n_experts,
                          int32_t hidden, int32_t inter, uint8_t *out, int32_t nthreads) {
    int64_t nb = (int64_t)hidden * inter / 256;
    int64_t mat_bytes = nb * 66, rec_bytes = 3 * mat_bytes;
    int64_t jobs = (int64_t)n_experts * 3;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t j = 0; j < jobs; j++) {
        int32_t e = (int32_t)(j / 3), m = (int32_t)(j % 3);
        synth_matrix_blocks(seed, layer, e0 + e, m, nb, out + (int64_t)e * rec_bytes + m * mat_bytes);
    }
}

/* n values ~ N(0, sigma^2), rounded to f32; value i is the cosine (i even) or sine
 * (i odd) half of one Box-Muller pair built from draws 2*(i/2) and 2*(i/2)+1. */
void synth_normal_f32(uint64_t seed, uint32_t tag, uint64_t a, uint64_t b, int64_t n,
                      double sigma, float *out, int32_t nthreads) {
    uint64_t key = synth_key(seed, tag, a, b);
    int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t p = 0; p < npairs; p++) {
        double u1 = unit_oc(draw(key, 2u * (uint64_t)p));
        double u2 = unit_co(draw(key, 2u * (uint64_t)p + 1u));
        double r = sqrt(-2.0 * synth_ln(u1)), sn, cs;
        synth_sincos2pi(u2, &sn, &cs);
        out[2 * p] = (float)(sigma * (r * cs));
        if (2 * p + 1 < n) out[2 * p + 1] = (float)(sigma * (r * sn));
    }
}

/* Fisher-Yates permutation of 0..n-1 driven by one stream. */
static void permute(uint64_t key, int32_t n, int32_t *perm) {
    for (int32_t i = 0; i < n; i++) perm[i] = i;
    for (int32_t i = n - 1; i > 0; i--) {
        uint32_t j = below(draw(key, (uint64_t)i), (uint32_t)i + 1u);
        int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
    }
}

/* Per-expert router bias of a Zipf(s) prior: a seeded permutation gives each expert a
 * rank 1..E and bias[e] = -s * ln(rank(e)) (log of the unnormalised prior). */
void synth_zipf_bias(uint64_t seed, int32_t layer, int32_t n_experts, double s, float *out,
                     int32_t *scratch_perm) {
    permute(synth_key(seed, TAG_ZIPF, (uint64_t)layer, 0), n_experts, scratch_perm);
    for (int32_t r = 0; r < n_experts; r++)
        out[scratch_perm[r]] = (float)(-s * synth_ln((double)(r + 1)));
}

/* Residency choice: a seeded permutation; its first n_res experts are resident (mask 1). */
void synth_resident_mask(uint64_t seed, int32_t layer, int32_t n_experts, int32_t n_res,
                         uint8_t *mask, int32_t *scratch_perm) {
    permute(synth_key(seed, TAG_RESID, (uint64_t)layer, 0), n_experts, scratch_perm);
    for (int32_t e = 0; e < n_experts; e++) mask[e] = 0;
    for (int32_t r = 0; r < n_res && r < n_experts; r++) mask[scratch_perm[r]] = 1;
}

/* Seeded permutation of 0..n-1 under its own tag/key (used to shuffle slot order). */
void synth_permutation(uint64_t seed, uint32_t tag, uint64_t a, int32_t n, int32_t *perm) {
    permute(synth_key(seed, tag, a, 0), n, perm);
}
