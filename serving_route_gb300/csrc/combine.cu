// combine.cu -- step 5 of the layer: the top-k weighted FP32 reduction of each
// token's routed FC2 rows, written as BF16 (flashinfer PR #4069, Description:
// "grouped combine with owner-side FP32 route reduction" followed by the BF16
// reduction; on one GPU the owner is the token itself, so the reduce is local).
//
// out[t, c] = bf16_rn( fma chain over active k = 0..K-1, ascending, of
//             w[t, k] * y[inv_pad[t*K + k], c] ), starting from +0.
// A token with no active route gets +0.  Masked weights (possibly NaN) are
// never read into the sum.  HBM-bound: each CTA streams its token's K rows of
// y with 16-byte loads and writes one 16-byte BF16 vector per thread step.
#include "common.cuh"
#include "internal.h"

namespace mm {

__global__ void __launch_bounds__(128) combine_kernel(const uint16_t* __restrict__ y,
                                                      const int32_t* __restrict__ inv_pad,
                                                      const float* __restrict__ w, int64_t T,
                                                      int K, int H, uint16_t* __restrict__ out) {
  __shared__ int32_t rows[8];
  __shared__ float wts[8];
  const int chunks = H >> 3;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < K) {
      rows[threadIdx.x] = inv_pad[t * K + threadIdx.x];
      wts[threadIdx.x] = w[t * K + threadIdx.x];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int k = 0; k < K; ++k) {
        const int32_t p = rows[k];
        if (p < 0) continue;
        const float wk = wts[k];
        const uint4 v = *reinterpret_cast<const uint4*>(y + (int64_t)p * H + c * 8);
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wk, bf16_bits_to_float(vv[i] & 0xFFFFu), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wk, bf16_bits_to_float(vv[i] >> 16), acc[2 * i + 1]);
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(out + t * H + c * 8) = o;
    }
  }
}

cudaError_t launch_combine(const Workspace& ws, const Layout& L, const float* topk_w,
                           uint16_t* out, int64_t T, cudaStream_t s) {
  int64_t grid = T < 152 * 32 ? T : 152 * 32;
  if (grid < 1) grid = 1;
  combine_kernel<<<(unsigned)grid, 128, 0, s>>>(ws.y, ws.inv_pad, topk_w, T, L.K, L.H, out);
  return cudaGetLastError();
}

}  // namespace mm
