/*
 * synth.c -- seeded, counter-based generator of synthetic inputs.
 *
 * This file only draws random numbers: it holds none of the frame-step
 * arithmetic.  Both the CUDA path (through its tests and bench) and the CPU
 * oracle receive the SAME host arrays produced here.
 *
 * Generator: Philox4x32-10, as published by Salmon, Moraes, Dror and Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3" (SC'11).  A 128-bit counter
 * (c0..c3) and a 64-bit key (k0,k1) go through ten rounds; each round
 * multiplies c0 and c2 by two fixed odd constants, mixes the high halves with
 * the other two words and the key, and the key is bumped by two Weyl
 * constants between rounds.  Element i of a stream is taken from the block
 * with counter (i/4 low word, i/4 high word, stream id, 0), word i%4, keyed
 * by the 64-bit seed.
 *
 * Normal deviates use the Box-Muller transform on two uniforms in (0,1);
 * integers in [lo,hi) use the multiply-shift reduction of a 32-bit word.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static void philox_block(const uint32_t in_ctr[4], const uint32_t in_key[2], uint32_t out[4])
{
    uint32_t c0 = in_ctr[0], c1 = in_ctr[1], c2 = in_ctr[2], c3 = in_ctr[3];
    uint32_t k0 = in_key[0], k1 = in_key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += PHILOX_W0; k1 += PHILOX_W1; }
        uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Raw access for known-answer tests. */
void synth_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    philox_block(ctr, key, out);
}

static void stream_block(uint64_t seed, uint32_t stream, uint64_t block, uint32_t out[4])
{
    uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), stream, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    philox_block(ctr, key, out);
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs only). */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* uniform in (0,1) from the top 24 bits of a word */
static float u01(uint32_t w) { return ((float)(w >> 8) + 0.5f) * (1.0f / 16777216.0f); }

/* four normals from one Philox block (two Box-Muller pairs) */
static void block_normals(const uint32_t w[4], float z[4])
{
    const float two_pi = 6.2831853071795864769f;
    for (int h = 0; h < 2; ++h) {
        float r = sqrtf(-2.0f * logf(u01(w[2 * h])));
        float a = two_pi * u01(w[2 * h + 1]);
        z[2 * h] = r * cosf(a);
        z[2 * h + 1] = r * sinf(a);
    }
}

/* Elements [offset, offset+n) of stream (seed, stream): N(mean, std) in fp32. */
void synth_normal_f32(uint64_t seed, uint32_t stream, uint64_t offset, int64_t n,
                      float mean, float std, float* out)
{
    if (n <= 0) return;
    uint64_t b0 = offset / 4, b1 = (offset + (uint64_t)n + 3) / 4;
#pragma omp parallel for schedule(static)
    for (int64_t b = (int64_t)b0; b < (int64_t)b1; ++b) {
        uint32_t w[4];
        float z[4];
        stream_block(seed, stream, (uint64_t)b, w);
        block_normals(w, z);
        for (int e = 0; e < 4; ++e) {
            uint64_t i = (uint64_t)b * 4 + (uint64_t)e;
            if (i < offset || i >= offset + (uint64_t)n) continue;
            out[i - offset] = mean + std * z[e];
        }
    }
}

/* Same draws, rounded to bf16 (round to nearest even); bits written as uint16. */
void synth_normal_bf16(uint64_t seed, uint32_t stream, uint64_t offset, int64_t n,
                       float mean, float std, uint16_t* out)
{
    if (n <= 0) return;
    uint64_t b0 = offset / 4, b1 = (offset + (uint64_t)n + 3) / 4;
#pragma omp parallel for schedule(static)
    for (int64_t b = (int64_t)b0; b < (int64_t)b1; ++b) {
        uint32_t w[4];
        float z[4];
        stream_block(seed, stream, (uint64_t)b, w);
        block_normals(w, z);
        for (int e = 0; e < 4; ++e) {
            uint64_t i = (uint64_t)b * 4 + (uint64_t)e;
            if (i < offset || i >= offset + (uint64_t)n) continue;
            out[i - offset] = f32_to_bf16_rne(mean + std * z[e]);
        }
    }
}

/* Integers uniform in [lo, hi) (hi > lo), by multiply-shift of a 32-bit word. */
void synth_uniform_int(uint64_t seed, uint32_t stream, uint64_t offset, int64_t n,
                       int32_t lo, int32_t hi, int32_t* out)
{
    if (n <= 0 || hi <= lo) return;
    uint64_t range = (uint64_t)((int64_t)hi - (int64_t)lo);
    uint64_t b0 = offset / 4, b1 = (offset + (uint64_t)n + 3) / 4;
#pragma omp parallel for schedule(static)
    for (int64_t b = (int64_t)b0; b < (int64_t)b1; ++b) {
        uint32_t w[4];
        stream_block(seed, stream, (uint64_t)b, w);
        for (int e = 0; e < 4; ++e) {
            uint64_t i = (uint64_t)b * 4 + (uint64_t)e;
            if (i < offset || i >= offset + (uint64_t)n) continue;
            out[i - offset] = lo + (int32_t)(((uint64_t)w[e] * range) >> 32);
        }
    }
}

/* bf16 bits -> fp32 values (exact), for host-side inspection in tests. */
void synth_bf16_to_f32(const uint16_t* in, int64_t n, float* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = (uint32_t)in[i] << 16;
        memcpy(&out[i], &u, 4);
    }
}
