/*
 * qdsynth — seeded synthetic inputs for the quantized decode path.
 *
 * This file is the ONE piece of code shared by the CUDA path's tests/bench and
 * the CPU oracle's tests: it produces bytes and numbers, and holds none of the
 * method's arithmetic (no dequantisation, no dot products, no norms).
 *
 * Generator: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  SplitMix64 is a counter-based
 * generator: the i-th output (0-based) of a stream whose state starts at s is
 *     mix64(s + (i + 1) * GAMMA),  GAMMA = 0x9E3779B97F4A7C15,
 * with the published 64-bit finaliser mix64.  Any element can therefore be
 * produced independently of the others, which lets tests regenerate a small
 * slice of a multi-gigabyte tensor, and lets the fill loops run in parallel.
 *
 * A stream is named: its start state is mix64(seed) XOR fnv1a64(name), so that
 * every tensor of a synthetic model gets its own reproducible stream.
 *
 * Uniform doubles in [0,1) take the top 53 bits.  Normals use the Box-Muller
 * transform (G. E. P. Box, M. E. Muller, 1958) on the consecutive uniform pair
 * (2p, 2p+1): r = sqrt(-2 ln(1-u0)), t = 2*pi*u1, outputs r cos t, r sin t.
 *
 * Portable C99 (plus optional OpenMP); no architecture intrinsics.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define QS_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t qs_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* FNV-1a, 64-bit (Fowler, Noll, Vo). */
static uint64_t qs_fnv1a64(const char* s) {
    uint64_t h = 0xCBF29CE484222325ULL;
    for (; s && *s; ++s) {
        h ^= (uint8_t)(*s);
        h *= 0x100000001B3ULL;
    }
    return h;
}

uint64_t qs_stream(uint64_t seed, const char* name) {
    return qs_mix64(seed) ^ qs_fnv1a64(name);
}

static inline uint64_t qs_at(uint64_t key, uint64_t i) {
    return qs_mix64(key + (i + 1) * QS_GAMMA);
}

static inline double qs_u01(uint64_t key, uint64_t i) {
    return (double)(qs_at(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

void qs_fill_u64(uint64_t key, uint64_t i0, int64_t n, uint64_t* out) {
#pragma omp parallel for schedule(static) if (n > 65536)
    for (int64_t i = 0; i < n; ++i) out[i] = qs_at(key, i0 + (uint64_t)i);
}

void qs_fill_uniform_f64(uint64_t key, uint64_t i0, int64_t n, double lo, double hi, double* out) {
#pragma omp parallel for schedule(static) if (n > 65536)
    for (int64_t i = 0; i < n; ++i) out[i] = lo + (hi - lo) * qs_u01(key, i0 + (uint64_t)i);
}

void qs_fill_uniform_f32(uint64_t key, uint64_t i0, int64_t n, double lo, double hi, float* out) {
#pragma omp parallel for schedule(static) if (n > 65536)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * qs_u01(key, i0 + (uint64_t)i));
}

/* Integers uniform on [lo, hi] (inclusive), written as int32. */
void qs_fill_int_i32(uint64_t key, uint64_t i0, int64_t n, int64_t lo, int64_t hi, int32_t* out) {
    const double span = (double)(hi - lo + 1);
#pragma omp parallel for schedule(static) if (n > 65536)
    for (int64_t i = 0; i < n; ++i) {
        int64_t v = lo + (int64_t)(qs_u01(key, i0 + (uint64_t)i) * span);
        if (v > hi) v = hi;
        out[i] = (int32_t)v;
    }
}

/* Integers uniform on [lo, hi] (inclusive, within -128..255), written as bytes
 * (two's complement for negative values). */
void qs_fill_int_u8(uint64_t key, uint64_t i0, int64_t n, int64_t lo, int64_t hi, uint8_t* out) {
    const double span = (double)(hi - lo + 1);
#pragma omp parallel for schedule(static) if (n > 65536)
    for (int64_t i = 0; i < n; ++i) {
        int64_t v = lo + (int64_t)(qs_u01(key, i0 + (uint64_t)i) * span);
        if (v > hi) v = hi;
        out[i] = (uint8_t)(v & 0xFF);
    }
}

/* Standard normals (Box-Muller), rounded to float.  Element i is member
 * (i & 1) of pair p = i >> 1, which uses uniforms 2p and 2p+1 of the stream. */
void qs_fill_normal_f32(uint64_t key, uint64_t i0, int64_t n, float* out) {
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static) if (n > 16384)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t e = i0 + (uint64_t)i;
        uint64_t p = e >> 1;
        double u0 = qs_u01(key, 2 * p);
        double u1 = qs_u01(key, 2 * p + 1);
        double r = sqrt(-2.0 * log(1.0 - u0));
        double t = two_pi * u1;
        out[i] = (float)((e & 1) ? r * sin(t) : r * cos(t));
    }
}

int qs_abi_version(void) { return 1; }
