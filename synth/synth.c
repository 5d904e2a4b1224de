/*
 * Seeded synthetic input generator, shared by the CPU oracle and the CUDA path.
 *
 * It holds none of the decode step's arithmetic: it only turns (seed, stream,
 * index) into numbers.  Every value is a pure function of those three, so any
 * slice of a tensor can be regenerated independently and the result does not
 * depend on the thread count.
 *
 * Counter-based generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11), written here from its
 * published definition: a 4x32-bit counter, a 2x32-bit key, ten rounds of two
 * 32x32->64 multiplies with the constants 0xD2511F53 / 0xCD9E8D57, and a Weyl
 * key schedule with 0x9E3779B9 / 0xBB67AE85.
 *
 * Counter layout: (element_pair_index lo, hi, stream lo, stream hi).
 * Key: (seed lo, seed hi).
 *
 * Normals: Box-Muller on two 53-bit uniforms in (0, 1).  Pair i gives elements
 * 2i (cosine branch) and 2i+1 (sine branch).  A value is rounded to fp32 (round
 * to nearest even) and, for bf16 outputs, then to bf16 (round to nearest even):
 * that two-step rounding is part of the input definition.
 *
 * Integers in [lo, hi): Lemire's multiply-shift on the first 32-bit word of
 * Philox(counter = (i, 0, stream)), a tiny bias that does not matter here.
 */
#define _GNU_SOURCE
#include <stdint.h>
#include <string.h>
#include <math.h>

typedef struct { uint32_t v[4]; } ph_ctr;

static ph_ctr philox4x32_10(ph_ctr c, uint32_t k0, uint32_t k1) {
    uint32_t c0 = c.v[0], c1 = c.v[1], c2 = c.v[2], c3 = c.v[3];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c1 = (uint32_t)p1;
        c3 = (uint32_t)p0;
        c0 = n0;
        c2 = n2;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    ph_ctr out = {{c0, c1, c2, c3}};
    return out;
}

static inline ph_ctr draw(uint64_t seed, uint64_t stream, uint64_t idx) {
    ph_ctr c;
    c.v[0] = (uint32_t)idx;
    c.v[1] = (uint32_t)(idx >> 32);
    c.v[2] = (uint32_t)stream;
    c.v[3] = (uint32_t)(stream >> 32);
    return philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
}

/* 53-bit uniform strictly inside (0, 1) from two 32-bit words. */
static inline double u53(uint32_t a, uint32_t b) {
    uint64_t m = ((uint64_t)(a >> 5) << 26) | (uint64_t)(b >> 6);
    return ((double)m + 0.5) * (1.0 / 9007199254740992.0);
}

static inline void normal_pair(uint64_t seed, uint64_t stream, uint64_t pair,
                               double* z0, double* z1) {
    ph_ctr r = draw(seed, stream, pair);
    double u1 = u53(r.v[0], r.v[1]);
    double u2 = u53(r.v[2], r.v[3]);
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586476925286766559 * u2;
    double c, s;
    sincos(ang, &s, &c);
    *z0 = rad * c;
    *z1 = rad * s;
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, double mean, double std,
                      float* out, int64_t n) {
    int64_t npair = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npair; ++p) {
        double z0, z1;
        normal_pair(seed, stream, (uint64_t)p, &z0, &z1);
        int64_t i = 2 * p;
        out[i] = (float)(mean + std * z0);
        if (i + 1 < n) out[i + 1] = (float)(mean + std * z1);
    }
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, double mean, double std,
                       uint16_t* out, int64_t n) {
    int64_t npair = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npair; ++p) {
        double z0, z1;
        normal_pair(seed, stream, (uint64_t)p, &z0, &z1);
        int64_t i = 2 * p;
        out[i] = f32_to_bf16_rne((float)(mean + std * z0));
        if (i + 1 < n) out[i + 1] = f32_to_bf16_rne((float)(mean + std * z1));
    }
}

/* Same as synth_normal_bf16 but the output has a row stride: rows of `cols`
 * elements are generated as one flat tensor of rows*cols values and written to
 * out[r*ld + c].  Used to place a [len][D] tensor inside a [maxpos][D] buffer. */
void synth_normal_bf16_strided(uint64_t seed, uint64_t stream, double mean, double std,
                               uint16_t* out, int64_t rows, int64_t cols, int64_t ld) {
    int64_t n = rows * cols;
    int64_t npair = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npair; ++p) {
        double z0, z1;
        normal_pair(seed, stream, (uint64_t)p, &z0, &z1);
        int64_t i = 2 * p;
        out[(i / cols) * ld + (i % cols)] = f32_to_bf16_rne((float)(mean + std * z0));
        if (i + 1 < n) out[((i + 1) / cols) * ld + ((i + 1) % cols)] = f32_to_bf16_rne((float)(mean + std * z1));
    }
}

void synth_uniform_int(uint64_t seed, uint64_t stream, int32_t lo, int32_t hi,
                       int32_t* out, int64_t n) {
    uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        ph_ctr r = draw(seed, stream, (uint64_t)i);
        out[i] = lo + (int32_t)(((uint64_t)r.v[0] * span) >> 32);
    }
}

/* Raw 32-bit words, for tests of the generator itself. */
void synth_raw_u32(uint64_t seed, uint64_t stream, uint64_t idx, uint32_t out[4]) {
    ph_ctr r = draw(seed, stream, idx);
    memcpy(out, r.v, sizeof(r.v));
}
