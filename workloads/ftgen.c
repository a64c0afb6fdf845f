/*
 * ftgen.c -- seeded synthetic inputs for the sparse-MoE layer step.
 *
 * This module holds no MoE arithmetic: no routing, no quantisation, no FFN.
 * It only turns (seed, stream, index) into numbers, so that the CUDA path's
 * tests and benchmark and the CPU oracle can be fed identical inputs.
 *
 * Generator: Philox4x32-10, the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11),
 * section 4 (multiplication-based S-box, 10 rounds, Weyl key schedule).
 * Normal variates: the Box-Muller transform (Box and Muller, 1958), evaluated
 * in fp64 and rounded once to fp32.
 *
 * Stream layout (all generators): counter = (q_lo, q_hi, stream_lo, stream_hi),
 * key = (seed_lo, seed_hi), where q indexes a Philox block.  One block gives
 * four 32-bit words: two 53-bit uniforms, i.e. one Box-Muller pair, so normal
 * element i of a stream comes from block q = i / 2 (cosine branch for even i,
 * sine branch for odd i), and uniform element i from block q = i / 2 as well.
 *
 * The CUDA library carries its own implementation of the same published
 * definition for weight tensors too large to generate on the host; the
 * known-answer vectors of the reference Philox implementation pin both.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define FTGEN_API __attribute__((visibility("default")))

static void philox_round(uint32_t c[4], const uint32_t k[2]) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c[1] ^ k[0];
    const uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

FTGEN_API void ftgen_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k[0] += 0x9E3779B9u;
            k[1] += 0xBB67AE85u;
        }
        philox_round(c, k);
    }
    memcpy(out, c, sizeof c);
}

static void block_words(uint64_t seed, uint64_t stream, uint64_t q, uint32_t w[4]) {
    const uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), (uint32_t)stream, (uint32_t)(stream >> 32)};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    ftgen_philox4x32_10(ctr, key, w);
}

/* 53-bit uniform from two words, in [0, 1). */
static double u53(uint32_t a, uint32_t b) {
    const uint64_t m = ((uint64_t)(a >> 5) << 26) | (uint64_t)(b >> 6);
    return (double)m * 0x1.0p-53;
}

/* Uniform element i in [0, 1): the first 53-bit uniform of block i/2 for even i, the second for odd i. */
FTGEN_API void ftgen_uniform_f64(uint64_t seed, uint64_t stream, uint64_t first, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
        const uint64_t i = first + (uint64_t)j;
        uint32_t w[4];
        block_words(seed, stream, i >> 1, w);
        out[j] = (i & 1) ? u53(w[2], w[3]) : u53(w[0], w[1]);
    }
}

/* Standard normal element i in fp64 (before any scaling). */
static double normal_at(uint64_t seed, uint64_t stream, uint64_t i) {
    uint32_t w[4];
    block_words(seed, stream, i >> 1, w);
    const double u1 = u53(w[0], w[1]) + 0x1.0p-53; /* (0, 1] so that log() is finite */
    const double u2 = u53(w[2], w[3]);             /* [0, 1) */
    const double rad = sqrt(-2.0 * log(u1));
    const double th = 6.283185307179586 * u2;
    return (i & 1) ? rad * sin(th) : rad * cos(th);
}

/* out[j] = (float)(sigma * Z_{first+j}), one rounding from fp64. */
FTGEN_API void ftgen_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, int64_t n, double sigma, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = (float)(sigma * normal_at(seed, stream, first + (uint64_t)j));
}

FTGEN_API void ftgen_normal_f64(uint64_t seed, uint64_t stream, uint64_t first, int64_t n, double sigma, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = sigma * normal_at(seed, stream, first + (uint64_t)j);
}

/* fp32 -> bf16 bit pattern, round to nearest even (inputs are finite). */
static uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* Activations: bf16 bits of round(sigma * Z). */
FTGEN_API void ftgen_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, int64_t n, double sigma, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
        const float f = (float)(sigma * normal_at(seed, stream, first + (uint64_t)j));
        out[j] = f32_to_bf16_bits(f);
    }
}
