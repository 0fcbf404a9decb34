/*
 * moegen.h -- seeded, counter-based synthetic input generator.
 *
 * This header is the one piece of code shared by the CPU oracle's inputs and
 * the GPU path's inputs.  It holds no arithmetic of the MoE layer itself: it
 * only turns (seed, stream, index) into bits.  The same definitions are
 * restated in numpy in gen/inputs.py; a test checks that the three
 * implementations (numpy, host C, CUDA) agree bit for bit.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used in counter form: output i of a stream
 * with key k is mix64(k + (i + 1) * GAMMA), which is exactly the i-th output of
 * a SplitMix64 state initialised to k.
 *
 * Normal variates: Irwin-Hall sum of twelve 16-bit uniforms (the four 16-bit
 * lanes of three consecutive 64-bit outputs), centred and scaled by 2^-16:
 *     z = (2*S - 12*65535) / 2^17,   S = sum of the twelve lanes.
 * Every step is an exact integer or power-of-two operation, so z is the same
 * IEEE float on every machine; mean 0, variance 1 - 2^-32, support (-6, 6).
 */
#ifndef MOEGEN_H
#define MOEGEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define MOEGEN_FN static __host__ __device__ __forceinline__
#else
#define MOEGEN_FN static inline
#endif

#define MOEGEN_GAMMA 0x9E3779B97F4A7C15ull

/* stream tags: one independent stream per synthetic tensor */
enum {
  MOEGEN_STREAM_X = 1,          /* activations x[t, j], index t*H + j          */
  MOEGEN_STREAM_W1 = 2,         /* W1[e, n, j], index (e*2I + n)*H + j          */
  MOEGEN_STREAM_W2 = 3,         /* W2[e, c, j], index (e*H + c)*I + j           */
  MOEGEN_STREAM_LOGITS = 4,     /* router logits [t, e], index t*E + e          */
  MOEGEN_STREAM_BLOCKPERM = 5,  /* block-permutation routing draws              */
  MOEGEN_STREAM_EXPERTPERM = 6, /* expert permutation of the skewed routing     */
  MOEGEN_STREAM_GUMBEL = 7,     /* Gumbel draws of the skewed routing           */
  MOEGEN_STREAM_WLOGITS = 8     /* logits of the K chosen experts, t*K + k      */
};

MOEGEN_FN uint64_t moegen_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* key of stream `tag` under `seed` */
MOEGEN_FN uint64_t moegen_key(uint64_t seed, uint64_t tag) {
  return moegen_mix64(seed * MOEGEN_GAMMA + tag);
}

/* i-th 64-bit output of the stream with key k */
MOEGEN_FN uint64_t moegen_u64(uint64_t key, uint64_t i) {
  return moegen_mix64(key + (i + 1ull) * MOEGEN_GAMMA);
}

MOEGEN_FN uint32_t moegen_lanesum(uint64_t v) {
  return (uint32_t)(v & 0xFFFFu) + (uint32_t)((v >> 16) & 0xFFFFu) +
         (uint32_t)((v >> 32) & 0xFFFFu) + (uint32_t)(v >> 48);
}

/* normal variate number j of the stream (consumes outputs 3j, 3j+1, 3j+2) */
MOEGEN_FN float moegen_normal(uint64_t key, uint64_t j) {
  uint32_t s = moegen_lanesum(moegen_u64(key, 3ull * j)) +
               moegen_lanesum(moegen_u64(key, 3ull * j + 1ull)) +
               moegen_lanesum(moegen_u64(key, 3ull * j + 2ull));
  int32_t c = 2 * (int32_t)s - 12 * 65535; /* |c| < 2^20: exact in float */
  return (float)c * (1.0f / 131072.0f);
}

/* bf16 bit pattern of a normal variate: the float's upper 16 bits
 * (truncation toward zero; a data recipe, not a rounding of the layer) */
MOEGEN_FN uint16_t moegen_normal_bf16_bits(uint64_t key, uint64_t j) {
  union { float f; uint32_t u; } v;
  v.f = moegen_normal(key, j);
  return (uint16_t)(v.u >> 16);
}

#endif /* MOEGEN_H */
