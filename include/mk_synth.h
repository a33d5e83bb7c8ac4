/*
 * mk_synth.h — seeded synthetic inputs for the decode megakernel: random-init
 * bf16 weights, token ids and stand-in KV-cache contents.
 *
 * This module holds none of the decoder's arithmetic. It exists so that the
 * GPU path and the CPU oracle can be fed bit-identical inputs without either
 * one producing the other's inputs: the host functions below fill host
 * memory, the device functions fill device memory, and both implement the
 * same counter-based generator from its published definition:
 *
 *   splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014; the 64-bit finaliser of java.util.SplittableRandom
 *   and of Vigna's splitmix64.c):
 *     mix(z) = let z1 = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                  z2 = (z1 ^ (z1 >> 27)) * 0x94D049BB133111EB
 *              in z2 ^ (z2 >> 31)
 *     the i-th output (i >= 0) of a stream whose state starts at s is
 *     mix(s + (i + 1) * 0x9E3779B97F4A7C15)            (all arithmetic mod 2^64)
 *
 * Streams used here:
 *   key(seed, tid)   = mix(seed + (tid + 1) * 0x9E3779B97F4A7C15)
 *   u(seed, tid, i)  = mix(key(seed, tid) + (i + 1) * 0x9E3779B97F4A7C15)
 *
 * Approximately normal values (Irwin-Hall of four 16-bit uniforms):
 *   S = sum of the four 16-bit fields of u            (integer in [0, 262140])
 *   z = (float)(S - 131070) * c                       (one fp32 multiply, RNE)
 *   c = (float)(sigma / sqrt(4 * (65536^2 - 1) / 12)) (exact variance sigma^2)
 *   value = bf16 round-to-nearest-even of (offset + z) (offset = 0 or 1, fp32 add)
 * (S - 131070) is an integer below 2^24, so it is exact in fp32, and the
 * result is bit-identical on any IEEE-754 machine.
 *
 * Token ids: tok = u(seed, tid, i) mod vocab.
 *
 * Tensor ids (tid) used by the tests and the bench are listed in
 * synth/__init__.py; any 64-bit value is accepted here.
 *
 * Errors: every function returns 0 on success, a negative value on invalid
 * arguments (null pointer, non-positive sizes) and, for device functions, a
 * positive cudaError_t value if the launch failed. Device functions are
 * asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 * default stream). All pointers are caller-owned.
 */
#ifndef MK_SYNTH_H
#define MK_SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The fp32 multiplier c for a target standard deviation sigma (see above). */
float mk_synth_scale(double sigma);

/* Raw splitmix64 stream: out[j] = mix(state + (i0 + j + 1) * 0x9E3779B97F4A7C15). */
int mk_synth_stream_host(uint64_t state, uint64_t i0, int64_t n, uint64_t *out);

/* Raw generator output u(seed, tid, i) for i in [i0, i0 + n) into out[n]. */
int mk_synth_u64_host(uint64_t seed, uint64_t tid, uint64_t i0, int64_t n, uint64_t *out);

/* out[j] = bf16(offset + z(u(seed, tid, i0 + j)) * c), j < n.  Host memory. */
int mk_synth_normal_bf16_host(uint16_t *out, int64_t n, uint64_t seed, uint64_t tid,
                              uint64_t i0, float c, float offset);

/* Same values, written to device memory by a CUDA kernel. */
int mk_synth_normal_bf16_device(uint16_t *out, int64_t n, uint64_t seed, uint64_t tid,
                                uint64_t i0, float c, float offset, void *stream);

/* tokens[j] = u(seed, tid, i0 + j) mod vocab, j < n.  Host memory. */
int mk_synth_tokens_host(int32_t *out, int64_t n, uint64_t seed, uint64_t tid,
                         uint64_t i0, int32_t vocab);

/* Stand-in paged KV-cache contents.  For batch row b, token t < ctx, kv head h
 * and dim e, the value is the normal generator at
 *   i = ((b * ctx + t) * n_kv_heads + h) * head_dim + e
 * of stream tid, written to pool[page_table[b*max_pages + t/page_size]]
 * [h][t % page_size][e] (pool layout [num_pages][n_kv_heads][page_size][head_dim],
 * one layer).  page_table is device memory for the device variant. */
int mk_synth_kv_pages_device(uint16_t *pool, const int32_t *page_table, int32_t batch,
                             int32_t max_pages, int32_t ctx, int32_t n_kv_heads,
                             int32_t page_size, int32_t head_dim, uint64_t seed,
                             uint64_t tid, float c, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MK_SYNTH_H */
