// combine.cu -- step 5 of the layer: the top-k weighted FP32 reduction of each
// token's routed FC2 rows, written as BF16 (flashinfer PR #4069, Description:
// the combine reduces each token's routes in FP32 on the owner and the result
// is reduced to BF16; on one GPU the owner is the token itself, so the reduce
// is local).
//
// out[t, c] = bf16_rn( fma chain over active k = 0..K-1, ascending, of
//             w[t, k] * y[inv_pad[t*K + k], c] ), starting from +0.
// A token with no active route gets +0.  Masked weights (possibly NaN) are
// never read into the sum.  HBM-bound: one thread owns 8 consecutive columns
// of one token, issues the K 16-byte loads of its routes together (masked
// routes read nothing), then folds them in ascending k; a CTA covers 1024
// columns of one token, so the grid spans tokens x column chunks.
#include "common.cuh"
#include "internal.h"

namespace mm {

constexpr int kCombineThreads = 128;
constexpr int kColsPerCta = kCombineThreads * 8;

template <int K>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const uint16_t* __restrict__ y, const int32_t* __restrict__ inv_pad,
    const float* __restrict__ w, int64_t T, int H, int col_ctas, uint16_t* __restrict__ out) {
  pdl_wait();
  const int64_t units = T * col_ctas;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t t = u / col_ctas;
    const int c = (int)(u - t * col_ctas) * kColsPerCta + threadIdx.x * 8;
    if (c >= H) continue;
    int32_t p[K];
    float wk[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      p[k] = __ldg(inv_pad + t * K + k);
      wk[k] = __ldg(w + t * K + k);
    }
    uint4 v[K];
#pragma unroll
    for (int k = 0; k < K; ++k)
      v[k] = (p[k] >= 0) ? *reinterpret_cast<const uint4*>(y + (int64_t)p[k] * H + c)
                         : make_uint4(0u, 0u, 0u, 0u);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (p[k] < 0) continue;
      const uint32_t vv[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(wk[k], bf16_bits_to_float(vv[i] & 0xFFFFu), acc[2 * i]);
        acc[2 * i + 1] = fmaf(wk[k], bf16_bits_to_float(vv[i] >> 16), acc[2 * i + 1]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(out + t * H + c) = o;
  }
  pdl_trigger();
}

template <int K>
static cudaError_t launch_k_combine(const Workspace& ws, const Layout& L, const float* topk_w,
                                   uint16_t* out, int64_t T, int col_ctas, unsigned grid,
                                   cudaStream_t s, bool pdl) {
  return launch_k(combine_kernel<K>, dim3(grid), dim3(kCombineThreads), 0, s, pdl, nullptr,
                  (const uint16_t*)ws.y, (const int32_t*)ws.inv_pad, topk_w, T, L.H, col_ctas, out);
}

cudaError_t launch_combine(const Workspace& ws, const Layout& L, const float* topk_w,
                           uint16_t* out, int64_t T, cudaStream_t s, bool pdl, int max_ctas) {
  const int col_ctas = (L.H + kColsPerCta - 1) / kColsPerCta;
  int64_t units = T * col_ctas;
  const int64_t cap = max_ctas;
  const unsigned grid = (unsigned)(units < cap ? (units < 1 ? 1 : units) : cap);
  switch (L.K) {
    case 1: return launch_k_combine<1>(ws, L, topk_w, out, T, col_ctas, grid, s, pdl);
    case 2: return launch_k_combine<2>(ws, L, topk_w, out, T, col_ctas, grid, s, pdl);
    case 4: return launch_k_combine<4>(ws, L, topk_w, out, T, col_ctas, grid, s, pdl);
    case 6: return launch_k_combine<6>(ws, L, topk_w, out, T, col_ctas, grid, s, pdl);
    case 8: return launch_k_combine<8>(ws, L, topk_w, out, T, col_ctas, grid, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mm
