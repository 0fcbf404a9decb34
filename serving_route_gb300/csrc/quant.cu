// quant.cu -- the element-wise kernels of the layer:
//   quant_dispatch  step 2 + 3: 1x128 FP8 E4M3 quantisation of x with a
//                   power-of-two scale per 128-column block ("DeepSeek-style
//                   FP8 block scaling", flashinfer PR #4069, Limitations),
//                   written straight into the padded, expert-sorted GEMM rows
//                   of every active route of the token (the dispatch gather
//                   fused into the quantiser: x is read once), in the blocked
//                   layout the GEMM loads (128x128 boxes).
//   swiglu_quant    the unfused reference path after FC1: SwiGLU of the BF16
//                   gate||up rows and 1x128 re-quantisation (flashinfer PR
//                   #4069, Description: the unfused path is the maintained
//                   reference, the fused epilogue must match it bit for bit).
//   quantize_weights / bind_transform: setup-time weight preparation (the
//                   blocked weight store and the GEMM scale atoms).
// All of them are HBM-bound streaming kernels: 16-byte loads, amax by
// shuffles, grids sized to the SM count.
#include "common.cuh"
#include "internal.h"

namespace mm {

__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// 8 floats -> 8 E4M3 codes with scale 2^e (v * 2^-e is exact).
__device__ __forceinline__ uint2 quant8(const float (&v)[8], int e) {
  const float inv = pow2_neg(e);
  uint2 q;
  q.x = e4m3x4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
  q.y = e4m3x4(v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
  return q;
}

// 8 floats -> 8 E4M3 codes of v * r (the per-tensor rule: one float product,
// then round to nearest even, saturating).
__device__ __forceinline__ uint2 quant8_rcp(const float (&v)[8], float r) {
  uint2 q;
  q.x = e4m3x4(__fmul_rn(v[0], r), __fmul_rn(v[1], r), __fmul_rn(v[2], r), __fmul_rn(v[3], r));
  q.y = e4m3x4(__fmul_rn(v[4], r), __fmul_rn(v[5], r), __fmul_rn(v[6], r), __fmul_rn(v[7], r));
  return q;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 p, float (&v)[8]) {
  const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
    v[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}

// One warp handles four 128-column blocks of one token per unit: eight lanes
// per block, each lane owning 16 consecutive columns (two 16-byte loads, one
// 16-byte store per route).  Each pass processes B units whose loads are
// issued together, so every warp keeps B KB of reads in flight, and each
// store instruction of the warp writes four whole 128-byte lines.
__device__ __forceinline__ float group8_max(float v) {
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// FMT 0: one power-of-two scale per 128 columns; 1 (MXFP8): one per 32
// columns (a lane pair); 2 (per-tensor): the static scale's float reciprocal
// rx for every value, block scales 1.
template <int FMT>
__device__ __forceinline__ void quant_dispatch_unit(const uint4 (&raw)[2], bool valid, int p_lane,
                                                    int b, int H, int K, int l8, float rx,
                                                    uint8_t* __restrict__ a,
                                                    uint8_t* __restrict__ a_sf) {
  constexpr bool MX = FMT == 1;
  float v[16];
  if (valid) {
    float lo[8], hi[8];
    unpack_bf16x8(raw[0], lo);
    unpack_bf16x8(raw[1], hi);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = lo[i];
      v[8 + i] = hi[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f;
  }
  int e = 0;
  float inv = rx;
  if (FMT != 2) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = MX ? fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1)) : group8_max(amax);
    e = pow2_scale_exp(amax);
    inv = pow2_neg(e);
  }
  uint4 q;
  q.x = e4m3x4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
  q.y = e4m3x4(v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
  q.z = e4m3x4(v[8] * inv, v[9] * inv, v[10] * inv, v[11] * inv);
  q.w = e4m3x4(v[12] * inv, v[13] * inv, v[14] * inv, v[15] * inv);
  const int KB = H >> 7;
  for (int k = 0; k < K; ++k) {
    const int p = __shfl_sync(0xFFFFFFFFu, p_lane, k);
    if (p >= 0 && valid) {
      *reinterpret_cast<uint4*>(a + blocked_offset(p, b * 128 + l8 * 16, H)) = q;
      if (MX) {
        // scale unit = 32-wide chunk 4b + l8/2 of the row
        if ((l8 & 1) == 0) a_sf[sf_atom_offset(p, 4 * b + (l8 >> 1), 4 * KB)] = (uint8_t)(e + 127);
      } else if (l8 == 0) {
        a_sf[sf_atom_offset(p, b, KB)] = (uint8_t)(e + 127);
      }
    }
  }
}

// B = 2: two units per pass, one unit per warp while the grid is not capped.
// B = 4: four units per pass at 64 registers (four blocks per SM), for a grid
// that then fits in one wave.
template <int FMT, int B>
__global__ void __launch_bounds__(256, B == 4 ? 4 : 1) quant_dispatch_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ inv_pad, int64_t T, int H, int K,
    const float* __restrict__ pt_rx, uint8_t* __restrict__ a, uint8_t* __restrict__ a_sf) {
  const int lane = threadIdx.x & 31, grp = lane >> 3, l8 = lane & 7;
  const int KB = H >> 7;
  const int units = (KB + 3) >> 2;
  const int64_t total = T * units;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  // x is an input of the forward that no kernel of it writes: a warp issues
  // the loads of its first pass before the programmatic wait, so their
  // latency overlaps the routing kernel's tail.  When every warp's work is
  // that one pass and the grid is one wave, nothing is left to load after
  // the routing ends.  The routing tables (inv_pad) and every store come
  // after the wait.
  bool waited = false;
  for (int64_t u0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u0 < total;
       u0 += B * nwarps) {
    uint4 r[B][2];
    int t[B];  // tokens fit in 32 bits: route ids t*K+k are int32
    int b[B];
    bool v[B];
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int64_t u = u0 + i * nwarps;
      const bool in = u < total;
      t[i] = in ? (int)(u / units) : 0;
      b[i] = in ? (int)(u - (int64_t)t[i] * units) * 4 + grp : KB;
      v[i] = b[i] < KB;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        r[i][h] = v[i] ? *reinterpret_cast<const uint4*>(x + (int64_t)t[i] * H + b[i] * 128 +
                                                         l8 * 16 + h * 8)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    // per-tensor: the static scale's reciprocal (written by
    // moe_set_activation_scales before any forward)
    const float rx = FMT == 2 ? *pt_rx : 1.0f;
    int p[B];
#pragma unroll
    for (int i = 0; i < B; ++i)
      p[i] = (lane < K && u0 + i * nwarps < total) ? inv_pad[(int64_t)t[i] * K + lane] : -1;
#pragma unroll
    for (int i = 0; i < B; ++i)
      quant_dispatch_unit<FMT>(r[i], v[i], p[i], b[i], H, K, l8, rx, a, a_sf);
  }
  pdl_trigger();
}

// Unfused SwiGLU + re-quantisation over the padded GEMM rows of this forward
// (MX: one scale per 32 columns, four lanes, instead of per 128).
template <int FMT>
__global__ void __launch_bounds__(256) swiglu_quant_kernel(
    const uint16_t* __restrict__ gu, const int32_t* __restrict__ total_mtiles, int I,
    const float* __restrict__ pt_rh, uint8_t* __restrict__ hq, uint8_t* __restrict__ h_sf) {
  constexpr bool MX = FMT == 1;
  pdl_wait();
  const float rh = FMT == 2 ? *pt_rh : 1.0f;
  const int lane = threadIdx.x & 31, half = lane >> 4, l16 = lane & 15;
  const int IB = I >> 7;
  const int units = (IB + 1) >> 1;
  const int64_t rows = (int64_t)(*total_mtiles) * 128;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < rows * units;
       u += nwarps) {
    const int64_t row = u / units;
    const int b = (int)(u - row * units) * 2 + half;
    const bool valid = b < IB;
    float g[8], up[8], h[8];
    if (valid) {
      const uint16_t* src = gu + row * 2 * I + b * 128 + l16 * 8;
      unpack_bf16x8(*reinterpret_cast<const uint4*>(src), g);
      unpack_bf16x8(*reinterpret_cast<const uint4*>(src + I), up);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = up[i] = 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      h[i] = swiglu(g[i], up[i]);
      amax = fmaxf(amax, fabsf(h[i]));
    }
    if (MX) {
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    } else {
      amax = half_warp_max(amax);
    }
    const int e = FMT == 2 ? 0 : pow2_scale_exp(amax);
    if (valid) {
      *reinterpret_cast<uint2*>(hq + blocked_offset(row, b * 128 + l16 * 8, I)) =
          FMT == 2 ? quant8_rcp(h, rh) : quant8(h, e);
      if (MX) {
        if ((l16 & 3) == 0) h_sf[sf_atom_offset(row, 4 * b + (l16 >> 2), 4 * IB)] = (uint8_t)(e + 127);
      } else if (l16 == 0) {
        h_sf[sf_atom_offset(row, b, IB)] = (uint8_t)(e + 127);
      }
    }
  }
  pdl_trigger();
}

// 128x128 block quantisation of float weights: one CTA per block, each thread
// owns half a row (64 floats in registers).
__global__ void __launch_bounds__(256) quantize_weights_kernel(const float* __restrict__ w,
                                                               int rows, int cols,
                                                               uint8_t* __restrict__ q,
                                                               float* __restrict__ scale) {
  __shared__ float red[8];
  const int rb = rows >> 7, cb = cols >> 7;
  const int64_t blk = blockIdx.x;
  const int64_t m = blk / ((int64_t)rb * cb);
  const int bi = (int)((blk / cb) % rb), bj = (int)(blk % cb);
  const int r = threadIdx.x >> 1, c0 = (threadIdx.x & 1) * 64;
  const int64_t base = (m * rows + (int64_t)bi * 128 + r) * cols + (int64_t)bj * 128 + c0;
  float v[64];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 f = *reinterpret_cast<const float4*>(w + base + 4 * i);
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const int e = pow2_scale_exp(amax);
  const float inv = pow2_neg(e);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 o;
    o.x = e4m3x4(v[16 * i + 0] * inv, v[16 * i + 1] * inv, v[16 * i + 2] * inv, v[16 * i + 3] * inv);
    o.y = e4m3x4(v[16 * i + 4] * inv, v[16 * i + 5] * inv, v[16 * i + 6] * inv, v[16 * i + 7] * inv);
    o.z = e4m3x4(v[16 * i + 8] * inv, v[16 * i + 9] * inv, v[16 * i + 10] * inv, v[16 * i + 11] * inv);
    o.w = e4m3x4(v[16 * i + 12] * inv, v[16 * i + 13] * inv, v[16 * i + 14] * inv, v[16 * i + 15] * inv);
    *reinterpret_cast<uint4*>(q + base + 16 * i) = o;
  }
  if (threadIdx.x == 0) scale[(m * rb + bi) * cb + bj] = pow2_neg(-e);
}

// NVFP4 checkpoint weights -> the 128x128 FP8 weight format (flashinfer PR
// #4069, Reviewer notes: NVFP4 checkpoints ride the FP8 backend unchanged
// through a one-time requantization).  An NVFP4 matrix holds E2M1 codes two
// per byte along the columns (the even column in the low nibble), an E4M3
// scale per 16 columns of a row and a float scale per matrix; each value is
// e2m1 * e4m3 * global with one float rounding (the first product is
// exact), then quantised as quantize_weights_kernel does.  The two decoders
// follow the formats' definitions.
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
  // sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0 is
  // the subnormal mantissa * 0.5
  const uint32_t e = (nib >> 1) & 3u, m = nib & 1u;
  const float mag =
      e == 0u ? 0.5f * (float)m : __int_as_float((int)((e + 126u) << 23)) * (1.0f + 0.5f * (float)m);
  return (nib & 8u) ? -mag : mag;
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  // OCP E4M3FN: exponent bits 6..3 (bias 7), mantissa bits 2..0; exponent 0
  // is the subnormal mantissa * 2^-9; S.1111.111 is NaN
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float mag;
  if (e == 15u && m == 7u)
    mag = __int_as_float(0x7FC00000);
  else if (e == 0u)
    mag = (float)m * 0.001953125f;
  else
    mag = __int_as_float((int)((e + 120u) << 23)) * (1.0f + 0.125f * (float)m);
  return (c & 0x80u) ? -mag : mag;
}

// One CTA per 128x128 block, a thread per half row (64 values: 32 code bytes,
// four block scales).
__global__ void __launch_bounds__(256) requant_nvfp4_kernel(const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ sblk,
                                                            const float* __restrict__ gs, int rows,
                                                            int cols, uint8_t* __restrict__ q,
                                                            float* __restrict__ scale) {
  __shared__ float red[8];
  const int rb = rows >> 7, cb = cols >> 7;
  const int64_t blk = blockIdx.x;
  const int64_t m = blk / ((int64_t)rb * cb);
  const int bi = (int)((blk / cb) % rb), bj = (int)(blk % cb);
  const int r = threadIdx.x >> 1, c0 = (threadIdx.x & 1) * 64;
  const int64_t row = m * rows + (int64_t)bi * 128 + r;
  const int64_t col = (int64_t)bj * 128 + c0;
  const float g = gs[m];
  const uint4 b0 = *reinterpret_cast<const uint4*>(codes + row * (cols / 2) + col / 2);
  const uint4 b1 = *reinterpret_cast<const uint4*>(codes + row * (cols / 2) + col / 2 + 16);
  const uint32_t sw = *reinterpret_cast<const uint32_t*>(sblk + row * (cols / 16) + col / 16);
  const uint32_t wd[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
  float v[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const uint32_t nib = (wd[i >> 3] >> (4 * (i & 7))) & 0xFu;
    const float sc = e4m3_value((sw >> (8 * (i >> 4))) & 0xFFu);
    v[i] = __fmul_rn(e2m1_value(nib) * sc, g);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const int e = pow2_scale_exp(amax);
  const float inv = pow2_neg(e);
  const int64_t base = row * cols + col;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 o;
    o.x = e4m3x4(v[16 * i + 0] * inv, v[16 * i + 1] * inv, v[16 * i + 2] * inv, v[16 * i + 3] * inv);
    o.y = e4m3x4(v[16 * i + 4] * inv, v[16 * i + 5] * inv, v[16 * i + 6] * inv, v[16 * i + 7] * inv);
    o.z = e4m3x4(v[16 * i + 8] * inv, v[16 * i + 9] * inv, v[16 * i + 10] * inv, v[16 * i + 11] * inv);
    o.w = e4m3x4(v[16 * i + 12] * inv, v[16 * i + 13] * inv, v[16 * i + 14] * inv, v[16 * i + 15] * inv);
    *reinterpret_cast<uint4*>(q + base + 16 * i) = o;
  }
  if (threadIdx.x == 0) scale[(m * rb + bi) * cb + bj] = pow2_neg(-e);
}

// MXFP8 weights: every row quantised in 1x32 blocks along its columns; one
// thread per 32-float chunk (chunks are contiguous, so the scale index is the
// chunk index: [nmat, rows, cols/32]).
__global__ void __launch_bounds__(256) quantize_weights_mx_kernel(const float* __restrict__ w,
                                                                  int64_t chunks,
                                                                  uint8_t* __restrict__ q,
                                                                  float* __restrict__ scale) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < chunks;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 f = *reinterpret_cast<const float4*>(w + i * 32 + 4 * k);
      v[4 * k] = f.x;
      v[4 * k + 1] = f.y;
      v[4 * k + 2] = f.z;
      v[4 * k + 3] = f.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
    const int e = pow2_scale_exp(amax);
    const float inv = pow2_neg(e);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 o;
      o.x = e4m3x4(v[16 * h + 0] * inv, v[16 * h + 1] * inv, v[16 * h + 2] * inv, v[16 * h + 3] * inv);
      o.y = e4m3x4(v[16 * h + 4] * inv, v[16 * h + 5] * inv, v[16 * h + 6] * inv, v[16 * h + 7] * inv);
      o.z = e4m3x4(v[16 * h + 8] * inv, v[16 * h + 9] * inv, v[16 * h + 10] * inv, v[16 * h + 11] * inv);
      o.w = e4m3x4(v[16 * h + 12] * inv, v[16 * h + 13] * inv, v[16 * h + 14] * inv, v[16 * h + 15] * inv);
      *reinterpret_cast<uint4*>(q + i * 32 + 16 * h) = o;
    }
    scale[i] = pow2_neg(-e);
  }
}

// float power-of-two scale -> E8M0 byte; anything else flags MOE_DEV_BAD_SCALE.
__device__ __forceinline__ uint8_t scale_to_e8m0(float s, uint32_t* status) {
  const uint32_t b = __float_as_uint(s);
  const uint32_t ef = (b >> 23) & 0xFFu, m = b & 0x7FFFFFu;
  if ((b >> 31) == 0u && m == 0u && ef >= 1u && ef <= 254u) return (uint8_t)ef;
  if (b == 0x00400000u) return 0;  // 2^-127
  record_status(status, MOE_DEV_BAD_SCALE);
  return 127;
}

// Bind-time weight layout: every 128-row x 128-column block of an expert's
// matrix is stored as one contiguous 16 KB box, [E][N/128][K/128][128][128],
// so a GEMM stage's weight box is one sequential DRAM read.  For W1 the
// rows are first re-ordered so that 256-row tile j is gate rows
// [128j, 128j+128) followed by up rows [128j, 128j+128) (one FC1 tile then
// owns whole 1x128 blocks of h).  One thread per 16-byte chunk.
__global__ void bind_blocked_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                   int E, int N, int K, int gate_up) {
  const int NB = N / 128, KB = K / 128;
  const int64_t total = (int64_t)E * N * (K / 16);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    // destination index -> (e, nb, kb, r, c)
    const int c = (int)(i & 7);
    const int r = (int)((i >> 3) & 127);
    const int64_t blk = i >> 10;  // (e * NB + nb) * KB + kb
    const int kb = (int)(blk % KB);
    const int64_t enb = blk / KB;
    const int nb = (int)(enb % NB);
    const int64_t e = enb / NB;
    int64_t n = (int64_t)nb * 128 + r;  // row of the (re-ordered) matrix
    if (gate_up) {
      const int I = N / 2;
      const int64_t j = n >> 8, within = n & 255;
      n = (within < 128) ? (j * 128 + within) : (I + j * 128 + within - 128);
    }
    reinterpret_cast<uint4*>(dst)[i] =
        *reinterpret_cast<const uint4*>(src + (e * N + n) * (int64_t)K + kb * 128 + c * 16);
  }
}

__global__ void bind_w1_scale_kernel(const float* __restrict__ s, uint8_t* __restrict__ d, int E,
                                     int IB, int HB, uint32_t* status) {
  const int64_t total = (int64_t)E * 2 * IB * HB;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / (2 * IB * HB), rem = i % (2 * IB * HB);
    const int64_t nb = rem / HB, kb = rem % HB;
    const int64_t src_nb = (nb & 1) ? (IB + (nb >> 1)) : (nb >> 1);
    d[i] = scale_to_e8m0(s[(e * 2 * IB + src_nb) * HB + kb], status);
  }
}

__global__ void scale_convert_kernel(const float* __restrict__ s, uint8_t* __restrict__ d,
                                     int64_t n, uint32_t* status) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    d[i] = scale_to_e8m0(s[i], status);
}

static int stream_grid(int64_t work, int per_block, int64_t cap = 152 * 16) {
  int64_t b = (work + per_block - 1) / per_block;
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

int quant_dispatch_resident(int fmt, int batch) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  const void* k4 = fmt == 2 ? (const void*)quant_dispatch_kernel<2, 4>
                            : (fmt == 1 ? (const void*)quant_dispatch_kernel<1, 4>
                                        : (const void*)quant_dispatch_kernel<0, 4>);
  const void* k2 = fmt == 2 ? (const void*)quant_dispatch_kernel<2, 2>
                            : (fmt == 1 ? (const void*)quant_dispatch_kernel<1, 2>
                                        : (const void*)quant_dispatch_kernel<0, 2>);
  const void* k = batch == 4 ? k4 : k2;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 256, 0) != cudaSuccess) return 0;
  return per_sm * sms;
}

cudaError_t launch_quant_dispatch(const Workspace& ws, const Layout& L, const uint16_t* x,
                                  int64_t T, cudaStream_t s, bool pdl, int max_ctas,
                                  int resident2, int resident4, const float* pt_rx) {
  // one unit = four 128-column blocks of a token, eight warps per block
  const int64_t units = T * ((L.H / 128 + 3) / 4);
  const int g2 = stream_grid(units, 8, max_ctas), g4 = stream_grid(units, 32, max_ctas);
  // four units per warp only where one unit per warp would take more than
  // one wave and four per warp fit in one
  const bool b4 = g2 > resident2 && g4 <= resident4 && g4 < max_ctas;
  const int fmt = L.pt ? 2 : (L.mx ? 1 : 0);
  if (b4) {
    auto k = fmt == 2 ? quant_dispatch_kernel<2, 4>
                      : (fmt == 1 ? quant_dispatch_kernel<1, 4> : quant_dispatch_kernel<0, 4>);
    return launch_k(k, dim3(g4), dim3(256), 0, s, pdl, nullptr, x, (const int32_t*)ws.inv_pad, T,
                    L.H, L.K, pt_rx, ws.a, ws.a_sf);
  }
  auto k = fmt == 2 ? quant_dispatch_kernel<2, 2>
                    : (fmt == 1 ? quant_dispatch_kernel<1, 2> : quant_dispatch_kernel<0, 2>);
  return launch_k(k, dim3(g2), dim3(256), 0, s, pdl, nullptr, x, (const int32_t*)ws.inv_pad, T,
                  L.H, L.K, pt_rx, ws.a, ws.a_sf);
}

cudaError_t launch_swiglu_quant(const Workspace& ws, const Layout& L, int max_ctas,
                                cudaStream_t s, bool pdl, const float* pt_rh) {
  const int64_t warps = (L.rows_alloc) * ((L.I / 128 + 1) / 2);
  auto k = L.pt ? swiglu_quant_kernel<2> : (L.mx ? swiglu_quant_kernel<1> : swiglu_quant_kernel<0>);
  return launch_k(k, dim3(stream_grid(warps, 8, max_ctas)), dim3(256), 0, s, pdl, nullptr,
                  (const uint16_t*)ws.gu, (const int32_t*)ws.total_mtiles, L.I, pt_rh, ws.hq,
                  ws.h_sf);
}

cudaError_t launch_quantize_weights(const float* w, int64_t nmat, int rows, int cols, uint8_t* q,
                                    float* scale, cudaStream_t s) {
  const int64_t blocks = nmat * (rows / 128) * (cols / 128);
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  quantize_weights_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, rows, cols, q, scale);
  return cudaGetLastError();
}

cudaError_t launch_requant_nvfp4(const uint8_t* codes, const uint8_t* sblk, const float* gs,
                                 int64_t nmat, int rows, int cols, uint8_t* q, float* scale,
                                 cudaStream_t s) {
  const int64_t blocks = nmat * (rows / 128) * (cols / 128);
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  requant_nvfp4_kernel<<<(unsigned)blocks, 256, 0, s>>>(codes, sblk, gs, rows, cols, q, scale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_weights_mx(const float* w, int64_t nmat, int rows, int cols, uint8_t* q,
                                       float* scale, cudaStream_t s) {
  const int64_t chunks = nmat * rows * (int64_t)(cols / 32);
  if (chunks == 0) return cudaSuccess;
  quantize_weights_mx_kernel<<<stream_grid(chunks, 256), 256, 0, s>>>(w, chunks, q, scale);
  return cudaGetLastError();
}

// MXFP8 weight-scale atoms: for every expert, 128-row block nb (W1 in the
// interleaved gate/up order of the weight store) and K block kb, one
// 512-byte atom; row r's word holds the E8M0 scales of its 32-wide chunks
// 4kb .. 4kb+3 (byte (r%32)*16 + (r/32)*4 + j).  One thread per word.
__global__ void sfb_atoms_mx_kernel(const float* __restrict__ sc, int E, int N, int KB, int gate_up,
                                    uint32_t* __restrict__ atoms, uint32_t* status) {
  const int NB = N / 128;
  const int64_t words = (int64_t)E * NB * KB * 128;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int wd = (int)(i & 127);
    const int64_t atom = i >> 7;
    const int kb = (int)(atom % KB);
    const int64_t enb = atom / KB;
    const int nb = (int)(enb % NB);
    const int64_t e = enb / NB;
    const int r = (wd & 3) * 32 + (wd >> 2);
    int64_t n = (int64_t)nb * 128 + r;  // row of the (re-ordered) matrix
    if (gate_up) {
      const int I = N / 2;
      const int64_t j = n >> 8, within = n & 255;
      n = (within < 128) ? (j * 128 + within) : (I + j * 128 + within - 128);
    }
    const float* src = sc + (e * N + n) * (int64_t)(4 * KB) + 4 * kb;
    uint32_t v = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) v |= (uint32_t)scale_to_e8m0(src[j], status) << (8 * j);
    atoms[i] = v;
  }
}

// Weight-scale atoms for the GEMM B operand: for every expert, 128-row block
// nb and group q of four K blocks, one 512-byte atom whose rows all hold the
// four E8M0 bytes sf[e][nb][4q .. 4q+3] (127, i.e. 2^0, past the last K
// block).  One thread per 32-bit word.
__global__ void sfb_atoms_kernel(const uint8_t* __restrict__ sf, int64_t nblocks, int KB,
                                 uint32_t* __restrict__ atoms) {
  const int KQ = (KB + 3) >> 2;
  const int64_t words = nblocks * KQ * 128;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t atom = i >> 7;
    const int64_t blk = atom / KQ;
    const int q = (int)(atom - blk * KQ);
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = 4 * q + j;
      const uint32_t v = kb < KB ? sf[blk * KB + kb] : 127u;
      w |= v << (8 * j);
    }
    atoms[i] = w;
  }
}

// Per-tensor weight quantisation (the per_tensor scale mode of flashinfer PR
// #4688): one scale per matrix, s = float(amax / 448) (1 for an all-zero
// matrix), codes = E4M3_RNE_sat(w * float(1 / s)).  Three passes over the
// caller's buffers, no scratch: the matrix amax is gathered as float bits in
// the scale array itself (non-negative floats order like their bits), then
// turned into the scale in place, then every value is encoded.
__global__ void pt_amax_kernel(const float* __restrict__ w, int64_t per_mat, int chunks_per_mat,
                               uint32_t* __restrict__ amax_bits) {
  const int64_t m = blockIdx.y;
  const float* src = w + m * per_mat;
  float amax = 0.f;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < per_mat;
       i += (int64_t)chunks_per_mat * blockDim.x * 4) {
    const float4 f = *reinterpret_cast<const float4*>(src + i);
    amax = fmaxf(fmaxf(amax, fabsf(f.x)), fmaxf(fmaxf(fabsf(f.y), fabsf(f.z)), fabsf(f.w)));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + m, __float_as_uint(amax));
}

__global__ void pt_scale_kernel(float* __restrict__ scale, int64_t nmat) {
  for (int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; m < nmat;
       m += (int64_t)gridDim.x * blockDim.x) {
    const float amax = scale[m];  // written as bits by pt_amax_kernel
    scale[m] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  }
}

__global__ void pt_quant_kernel(const float* __restrict__ w, int64_t per_mat,
                                const float* __restrict__ scale, uint8_t* __restrict__ q) {
  const int64_t m = blockIdx.y;
  const float r = __fdiv_rn(1.0f, scale[m]);
  const float* src = w + m * per_mat;
  uint8_t* dst = q + m * per_mat;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < per_mat;
       i += (int64_t)gridDim.x * blockDim.x * 8) {
    const float4 a = *reinterpret_cast<const float4*>(src + i);
    const float4 b = *reinterpret_cast<const float4*>(src + i + 4);
    uint2 o;
    o.x = e4m3x4(__fmul_rn(a.x, r), __fmul_rn(a.y, r), __fmul_rn(a.z, r), __fmul_rn(a.w, r));
    o.y = e4m3x4(__fmul_rn(b.x, r), __fmul_rn(b.y, r), __fmul_rn(b.z, r), __fmul_rn(b.w, r));
    *reinterpret_cast<uint2*>(dst + i) = o;
  }
}

cudaError_t launch_quantize_weights_pt(const float* w, int64_t nmat, int rows, int cols, uint8_t* q,
                                       float* scale, cudaStream_t s) {
  if (nmat == 0) return cudaSuccess;
  if (nmat > 65535) return cudaErrorInvalidValue;
  const int64_t per_mat = (int64_t)rows * cols;
  if (cudaMemsetAsync(scale, 0, sizeof(float) * nmat, s) != cudaSuccess) return cudaGetLastError();
  const int chunks = (int)((per_mat / 4 + 255) / 256 < 64 ? (per_mat / 4 + 255) / 256 : 64);
  pt_amax_kernel<<<dim3(chunks, (unsigned)nmat), 256, 0, s>>>(w, per_mat, chunks,
                                                              reinterpret_cast<uint32_t*>(scale));
  pt_scale_kernel<<<(unsigned)((nmat + 255) / 256), 256, 0, s>>>(scale, nmat);
  const int qchunks = (int)((per_mat / 8 + 255) / 256 < 512 ? (per_mat / 8 + 255) / 256 : 512);
  pt_quant_kernel<<<dim3(qchunks, (unsigned)nmat), 256, 0, s>>>(w, per_mat, scale, q);
  return cudaGetLastError();
}

// Per-tensor scales of a bound layer: the weight scales are copied at bind
// (each must be a positive finite float); the static activation scales come
// from moe_set_activation_scales, which also precomputes, per expert, the
// factors the GEMM epilogues apply to their FP32 accumulators (x_scale *
// s_w1[e] for FC1, h_scale * s_w2[e] for FC2) and the activation scales'
// float reciprocals the quantisers multiply by.
__global__ void pt_check_scales_kernel(const float* __restrict__ s, int n, float* __restrict__ dst,
                                       uint32_t* status) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float v = s[i];
    if (!(v > 0.f) || !isfinite(v)) record_status(status, MOE_DEV_BAD_SCALE);
    dst[i] = v;
  }
}

__global__ void pt_set_scales_kernel(float* __restrict__ pt, int E, float x_scale, float h_scale) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    pt[2 * E + e] = __fmul_rn(x_scale, pt[e]);      // FC1 factor
    pt[3 * E + e] = __fmul_rn(h_scale, pt[E + e]);  // FC2 factor
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    pt[4 * E] = __fdiv_rn(1.0f, x_scale);
    pt[4 * E + 1] = __fdiv_rn(1.0f, h_scale);
  }
}

cudaError_t launch_pt_set_scales(const WeightStore& wst, const Layout& L, float x_scale,
                                 float h_scale, cudaStream_t s) {
  pt_set_scales_kernel<<<(L.E + 255) / 256, 256, 0, s>>>(wst.pt, L.E, x_scale, h_scale);
  return cudaGetLastError();
}

cudaError_t launch_bind_transform(const WeightStore& wst, const Layout& L, const uint8_t* w1,
                                  const float* w1s, const uint8_t* w2, const float* w2s,
                                  uint32_t* status, cudaStream_t s) {
  const int E = L.E, I = L.I, H = L.H;
  const int64_t w1_chunks = (int64_t)E * 2 * I * (H / 16), w2_chunks = (int64_t)E * H * (I / 16);
  bind_blocked_kernel<<<stream_grid(w1_chunks, 256), 256, 0, s>>>(w1, wst.w1, E, 2 * I, H, 1);
  bind_blocked_kernel<<<stream_grid(w2_chunks, 256), 256, 0, s>>>(w2, wst.w2, E, H, I, 0);
  if (L.pt) {
    // per-tensor: every block scale the tensor core applies is 1 (E8M0 127);
    // the expert scales go to the epilogue factors
    const size_t sf1 = (size_t)E * (2 * I / 128) * (H / 128), sf2 = (size_t)E * (H / 128) * (I / 128);
    const size_t at1 = (size_t)E * (2 * I / 128) * ((H / 128 + 3) / 4) * kSfAtomBytes;
    const size_t at2 = (size_t)E * (H / 128) * ((I / 128 + 3) / 4) * kSfAtomBytes;
    if (cudaMemsetAsync(wst.w1_sf, 127, sf1, s) != cudaSuccess ||
        cudaMemsetAsync(wst.w2_sf, 127, sf2, s) != cudaSuccess ||
        cudaMemsetAsync(wst.w1_sfatoms, 127, at1, s) != cudaSuccess ||
        cudaMemsetAsync(wst.w2_sfatoms, 127, at2, s) != cudaSuccess)
      return cudaGetLastError();
    pt_check_scales_kernel<<<(E + 255) / 256, 256, 0, s>>>(w1s, E, wst.pt, status);
    pt_check_scales_kernel<<<(E + 255) / 256, 256, 0, s>>>(w2s, E, wst.pt + E, status);
    return cudaGetLastError();
  }
  if (L.mx) {
    const int64_t words1 = (int64_t)E * (2 * I / 128) * (H / 128) * 128;
    const int64_t words2 = (int64_t)E * (H / 128) * (I / 128) * 128;
    sfb_atoms_mx_kernel<<<stream_grid(words1, 256), 256, 0, s>>>(
        w1s, E, 2 * I, H / 128, 1, reinterpret_cast<uint32_t*>(wst.w1_sfatoms), status);
    sfb_atoms_mx_kernel<<<stream_grid(words2, 256), 256, 0, s>>>(
        w2s, E, H, I / 128, 0, reinterpret_cast<uint32_t*>(wst.w2_sfatoms), status);
    return cudaGetLastError();
  }
  const int64_t n1 = (int64_t)E * 2 * (I / 128) * (H / 128);
  bind_w1_scale_kernel<<<stream_grid(n1, 256), 256, 0, s>>>(w1s, wst.w1_sf, E, I / 128, H / 128,
                                                            status);
  const int64_t n2 = (int64_t)E * (H / 128) * (I / 128);
  scale_convert_kernel<<<stream_grid(n2, 256), 256, 0, s>>>(w2s, wst.w2_sf, n2, status);
  const int64_t nb1 = (int64_t)E * (2 * I / 128), nb2 = (int64_t)E * (H / 128);
  sfb_atoms_kernel<<<stream_grid(nb1 * ((H / 128 + 3) / 4) * 128, 256), 256, 0, s>>>(
      wst.w1_sf, nb1, H / 128, reinterpret_cast<uint32_t*>(wst.w1_sfatoms));
  sfb_atoms_kernel<<<stream_grid(nb2 * ((I / 128 + 3) / 4) * 128, 256), 256, 0, s>>>(
      wst.w2_sf, nb2, I / 128, reinterpret_cast<uint32_t*>(wst.w2_sfatoms));
  return cudaGetLastError();
}

}  // namespace mm
