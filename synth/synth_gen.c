/*
 * Seeded synthetic-input generator (weights, norm scales, prompt token ids).
 *
 * This file holds no arithmetic of the decoding method: it only turns
 * (seed, stream, index) into numbers.  Both the CPU oracle and the CUDA
 * library receive their inputs from it, so the two sides see identical
 * values without sharing any model code.
 *
 * Generator: Philox4x32-10, the counter-based generator published by
 * Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as
 * 1, 2, 3" (SC'11).  Element j of a stream is a pure function of
 * (seed, stream, j), so tensors can be produced in parallel and in any
 * order.  Normal deviates use the Box-Muller transform on two 53-bit
 * uniforms built from one Philox output block.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static inline void philox_round(uint32_t c[4], const uint32_t k[2]) {
    uint64_t p0 = (uint64_t)PHILOX_M0 * c[0];
    uint64_t p1 = (uint64_t)PHILOX_M1 * c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k[0];
    uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

/* Ten rounds; the key is bumped by the Weyl constants between rounds. */
void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t k[2] = {key_in[0], key_in[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k[0] += PHILOX_W0;
            k[1] += PHILOX_W1;
        }
        philox_round(c, k);
    }
    memcpy(out, c, sizeof(c));
}

static inline void block_for(uint64_t seed, uint32_t stream, uint32_t lane, uint64_t j, uint32_t out[4]) {
    uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), stream, lane};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    synth_philox4x32_10(ctr, key, out);
}

/* Normal deviates N(mean, std^2), rounded once from double to float.
 * Block j yields elements 2j and 2j+1. */
void synth_normal_f32(uint64_t seed, uint32_t stream, uint64_t n, double mean, double std, float* out) {
    const double two_pi = 6.283185307179586476925286766559;
    const double inv53 = 1.0 / 9007199254740992.0; /* 2^-53 */
    int64_t npairs = (int64_t)((n + 1) / 2);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < npairs; ++j) {
        uint32_t x[4];
        block_for(seed, stream, 0u, (uint64_t)j, x);
        uint64_t a = ((uint64_t)x[0] << 32) | x[1];
        uint64_t b = ((uint64_t)x[2] << 32) | x[3];
        double u1 = (double)((a >> 11) + 1) * inv53; /* (0, 1] */
        double u2 = (double)(b >> 11) * inv53;       /* [0, 1) */
        double r = sqrt(-2.0 * log(u1));
        double t = two_pi * u2;
        double z0 = r * cos(t), z1 = r * sin(t);
        uint64_t i0 = 2 * (uint64_t)j;
        out[i0] = (float)(mean + std * z0);
        if (i0 + 1 < n) out[i0 + 1] = (float)(mean + std * z1);
    }
}

/* Uniform integers in [0, range) by the multiply-shift map (x * range) >> 32.
 * Block j yields elements 4j .. 4j+3. */
void synth_uniform_i32(uint64_t seed, uint32_t stream, uint64_t n, uint32_t range, int32_t* out) {
    int64_t nblk = (int64_t)((n + 3) / 4);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nblk; ++j) {
        uint32_t x[4];
        block_for(seed, stream, 1u, (uint64_t)j, x);
        for (int e = 0; e < 4; ++e) {
            uint64_t i = 4 * (uint64_t)j + (uint64_t)e;
            if (i < n) out[i] = (int32_t)(((uint64_t)x[e] * range) >> 32);
        }
    }
}

/* float -> bfloat16 bit pattern, round to nearest even (finite inputs). */
void synth_f32_to_bf16(const float* in, uint16_t* out, uint64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < (int64_t)n; ++i) {
        uint32_t u;
        memcpy(&u, &in[i], 4);
        uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
        out[i] = (uint16_t)((u + bias) >> 16);
    }
}

/* bfloat16 bit pattern -> float (exact). */
void synth_bf16_to_f32(const uint16_t* in, float* out, uint64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < (int64_t)n; ++i) {
        uint32_t u = (uint32_t)in[i] << 16;
        memcpy(&out[i], &u, 4);
    }
}
