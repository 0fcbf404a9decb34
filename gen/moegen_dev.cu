/*
 * moegen_dev.cu -- the same counter-based generator (moegen.h) on the GPU, used
 * to create full-size synthetic weights and activations directly in HBM.
 * Nothing here is arithmetic of the MoE layer.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "moegen.h"

__global__ void moegen_normal_f32_kernel(uint64_t key, uint64_t offset, int64_t n, float sigma,
                                         float* __restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float z = moegen_normal(key, offset + (uint64_t)i);
    out[i] = __fmul_rn(z, sigma);
  }
}

__global__ void moegen_normal_bf16_kernel(uint64_t key, uint64_t offset, int64_t n,
                                          uint16_t* __restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = moegen_normal_bf16_bits(key, offset + (uint64_t)i);
}

static int grid_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  if (b > 152 * 32) b = 152 * 32;
  if (b < 1) b = 1;
  return (int)b;
}

extern "C" int moegen_dev_fill_normal_f32(uint64_t seed, uint32_t tag, uint64_t offset, int64_t n,
                                          float sigma, float* d_out, cudaStream_t stream) {
  if (n <= 0) return 0;
  moegen_normal_f32_kernel<<<grid_for(n), 256, 0, stream>>>(moegen_key(seed, tag), offset, n,
                                                            sigma, d_out);
  return (int)cudaGetLastError();
}

extern "C" int moegen_dev_fill_normal_bf16(uint64_t seed, uint32_t tag, uint64_t offset, int64_t n,
                                           uint16_t* d_out, cudaStream_t stream) {
  if (n <= 0) return 0;
  moegen_normal_bf16_kernel<<<grid_for(n), 256, 0, stream>>>(moegen_key(seed, tag), offset, n,
                                                             d_out);
  return (int)cudaGetLastError();
}
