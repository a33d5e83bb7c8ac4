/*
 * synth.c — host half of the seeded input generator (see include/mk_synth.h
 * for the definition).  Plain C, OpenMP over elements; every element is a
 * pure function of (seed, tid, index), so the thread split cannot change it.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "mk_synth.h"

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t sm_key(uint64_t seed, uint64_t tid) { return sm_mix(seed + (tid + 1) * GOLDEN); }

static inline uint64_t sm_u(uint64_t key, uint64_t i) { return sm_mix(key + (i + 1) * GOLDEN); }

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    /* Values here are finite; round half to even on the 16 dropped bits. */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline uint16_t normal_bf16(uint64_t u, float c, float offset) {
    int32_t s = (int32_t)(u & 0xFFFF) + (int32_t)((u >> 16) & 0xFFFF) + (int32_t)((u >> 32) & 0xFFFF) +
                (int32_t)(u >> 48);
    volatile float z = (float)(s - 131070) * c; /* one fp32 multiply, no contraction */
    float v = offset + z;
    return f32_to_bf16_rne(v);
}

float mk_synth_scale(double sigma) { return (float)(sigma / sqrt(4.0 * (65536.0 * 65536.0 - 1.0) / 12.0)); }

int mk_synth_stream_host(uint64_t state, uint64_t i0, int64_t n, uint64_t *out) {
    if (!out || n < 0) return -1;
    for (int64_t j = 0; j < n; ++j) out[j] = sm_u(state, i0 + (uint64_t)j);
    return 0;
}

int mk_synth_u64_host(uint64_t seed, uint64_t tid, uint64_t i0, int64_t n, uint64_t *out) {
    if (!out || n < 0) return -1;
    uint64_t key = sm_key(seed, tid);
    for (int64_t j = 0; j < n; ++j) out[j] = sm_u(key, i0 + (uint64_t)j);
    return 0;
}

int mk_synth_normal_bf16_host(uint16_t *out, int64_t n, uint64_t seed, uint64_t tid, uint64_t i0, float c,
                              float offset) {
    if (!out || n < 0) return -1;
    uint64_t key = sm_key(seed, tid);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = normal_bf16(sm_u(key, i0 + (uint64_t)j), c, offset);
    return 0;
}

int mk_synth_tokens_host(int32_t *out, int64_t n, uint64_t seed, uint64_t tid, uint64_t i0, int32_t vocab) {
    if (!out || n < 0 || vocab <= 0) return -1;
    uint64_t key = sm_key(seed, tid);
    for (int64_t j = 0; j < n; ++j) out[j] = (int32_t)(sm_u(key, i0 + (uint64_t)j) % (uint64_t)vocab);
    return 0;
}
