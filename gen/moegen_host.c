/*
 * moegen_host.c -- bulk host generation of the synthetic inputs (OpenMP).
 * Definitions live in moegen.h; nothing here is arithmetic of the MoE layer.
 */
#include <stddef.h>
#include <stdint.h>
#include "moegen.h"

/* out[i] = normal(offset + i) * sigma  (single float multiply, round to nearest) */
void moegen_fill_normal_f32(uint64_t seed, uint32_t tag, uint64_t offset, int64_t n,
                            float sigma, float* out) {
  const uint64_t key = moegen_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float z = moegen_normal(key, offset + (uint64_t)i);
    out[i] = z * sigma;
  }
}

/* out[i] = bf16 bits of normal(offset + i) */
void moegen_fill_normal_bf16(uint64_t seed, uint32_t tag, uint64_t offset, int64_t n,
                             uint16_t* out) {
  const uint64_t key = moegen_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = moegen_normal_bf16_bits(key, offset + (uint64_t)i);
}

/* raw 64-bit outputs (used by the numpy cross-check) */
void moegen_fill_u64(uint64_t seed, uint32_t tag, uint64_t offset, int64_t n, uint64_t* out) {
  const uint64_t key = moegen_key(seed, tag);
  for (int64_t i = 0; i < n; ++i) out[i] = moegen_u64(key, offset + (uint64_t)i);
}
