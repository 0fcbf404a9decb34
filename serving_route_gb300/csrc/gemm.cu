// gemm.cu -- steps 3 and 4 of the layer: the FC1 and FC2 grouped GEMMs over
// block-scaled FP8 expert weights (flashinfer PR #4069, Description: FC1 with
// fused SwiGLU + 1x128 quantization, then FC2; the DeepGEMM WGMMA kernels of
// that page are prior art for Hopper, not the design used here).
//
// GB300 design:
//  * tcgen05.mma kind::mxf8f6f4 with block scales: both operands E4M3, one
//    E8M0 scale per row per 32-wide K chunk.  Every scale of the layer is a
//    power of two, so a 1x128 activation scale is four equal E8M0 bytes and a
//    128x128 weight scale is one byte for 128 rows; the tensor core applies
//    them exactly while it accumulates in FP32 in tensor memory.  No
//    per-K-block promotion through registers is needed.
//  * Persistent CTAs (one per SM) walk a static tile list: 128 padded rows of
//    one expert x 256 output columns, expert-major, so the two-or-more
//    m-tiles sharing a weight tile run at the same time and hit it in L2.
//    The tile count and the m-tile -> expert table come from device memory:
//    no host synchronisation, graph-capturable.
//  * Warp roles (192 threads): warp 0 feeds a 4-stage shared-memory ring with
//    TMA (A 128x128 B, B 256x128 B, 128-byte swizzle) plus a bulk copy of the
//    A scale atom; it writes the B scale atoms itself.  One thread of warp 1
//    copies the atoms into TMEM (tcgen05.cp) and issues the MMAs.  Warps 2-5
//    drain the 128x256 FP32 accumulator from TMEM and run the epilogue.
//  * Epilogues: FC2 -> BF16 y; FC1 unfused -> BF16 gate||up; FC1 fused ->
//    BF16-rounded gate/up, SwiGLU, 1x128 re-quantisation to E4M3 + E8M0 atoms
//    (bit-equal to the unfused path, which runs the same device functions).
//  * Every wait is bounded (1 s); on expiry the kernel records
//    MOE_DEV_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

namespace mm {

constexpr int kStages = 4;
constexpr int kEpiWarps = 8;                       // two per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;      // producer, MMA, epilogue
constexpr uint32_t kOffA = 0;                    // 128 rows x 128 B
constexpr uint32_t kOffB = 16384;                // 256 rows x 128 B
constexpr uint32_t kOffSfa = 49152;              // one 512 B atom
constexpr uint32_t kOffSfb = 49664;              // two 512 B atoms
constexpr uint32_t kStageBytes = 51200;          // multiple of 1024
constexpr uint32_t kTxBytes = 16384 + 32768 + 512;
constexpr uint32_t kTmemCols = 512;
// Scale factors live in TMEM after the accumulator (columns 0-255): one
// 16-column slot per pipeline stage (A atom at +0, B atoms at +8 and +12), so
// the copy for stage s+1 never overwrites scales the MMAs of stage s still read.
constexpr uint32_t kColSf = 256, kSfSlotCols = 16;
// One M=128 x N=256 MMA per 32-wide K chunk (B scales of the two 128-row
// blocks in adjacent 4-column groups); false issues two N=128 MMAs instead.
constexpr bool kSingleN256 = true;
constexpr size_t kDynSmem = (size_t)kStages * kStageBytes + 1024;

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB, const GemmArgs g) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar, acce_bar, drain_bar;
  __shared__ __align__(8) uint64_t amax_bar[4];  // per quadrant: both column halves posted
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ uint8_t sfb_sm[2][2][128];
  __shared__ float amax_sh[2][2][128];  // [tile parity][column half][row] (fused epilogue)

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int mtiles = *g.total_mtiles;
  if (mtiles > g.max_mtiles) mtiles = g.max_mtiles;
  const int total = mtiles * g.NT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&accf_bar), 1);
    mbar_init(smem_u32(&acce_bar), kEpiWarps);
    mbar_init(smem_u32(&drain_bar), 1);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&amax_bar[i]), 2);
    abort_sh = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort = &abort_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per tile the producer needs the expert id (a global table) and the
    // tile's weight-scale bytes.  Both are fetched ahead: the expert id two
    // tiles ahead, the scale bytes one tile ahead, so no dependent global load
    // stalls the producer at a tile boundary.
    auto expert_of = [&](int tile) -> int {
      return tile < total ? g.mtile_expert[tile / g.NT] : 0;
    };
    uint32_t nb0[4], nb1[4];
    auto fetch_sfb = [&](int tile, int e) {
      if (tile < total) {
        const int nt = tile - (tile / g.NT) * g.NT;
        const uint8_t* p = g.sfb + ((int64_t)e * g.NB + 2 * nt) * g.KB;
        const bool has1 = 2 * nt + 1 < g.NB;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kb = lane + 32 * i;
          nb0[i] = (kb < g.KB) ? p[kb] : 127u;
          nb1[i] = (has1 && kb < g.KB) ? p[g.KB + kb] : 127u;
        }
      }
    };
    auto stash_sfb = [&](int buf) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sfb_sm[buf][0][lane + 32 * i] = (uint8_t)nb0[i];
        sfb_sm[buf][1][lane + 32 * i] = (uint8_t)nb1[i];
      }
      __syncwarp();
    };
    // weight rows of a tile: expert e, 256-row n-tile
    auto b_row = [&](int tile, int e) { return e * g.N + (tile - (tile / g.NT) * g.NT) * 256; };
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued at least once, parity of last issue
    int buf = 0;
    const int G = gridDim.x;
    int e_cur = expert_of(blockIdx.x);
    int e_next = expert_of(blockIdx.x + G);
    fetch_sfb(blockIdx.x, e_cur);
    stash_sfb(0);
    for (int tile = blockIdx.x; tile < total && !*abort; tile += G) {
      const int mt = tile / g.NT;
      const int e = e_cur;
      const int e_after = expert_of(tile + 2 * G);  // needed one tile from now
      fetch_sfb(tile + G, e_next);                  // consumed after this tile's k loop
      const int y_b = b_row(tile, e);
      bool ok = true;
      for (int kb = 0; kb < g.KB; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort, g.status)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + stage * kStageBytes;
        const uint32_t v0 = (uint32_t)sfb_sm[buf][0][kb] * 0x01010101u;
        const uint32_t v1 = (uint32_t)sfb_sm[buf][1][kb] * 0x01010101u;
        *reinterpret_cast<uint4*>(st + kOffSfb + lane * 16) = make_uint4(v0, v0, v0, v0);
        *reinterpret_cast<uint4*>(st + kOffSfb + 512 + lane * 16) = make_uint4(v1, v1, v1, v1);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const uint32_t fb = smem_u32(&full_bar[stage]);
          const uint32_t sst = sbase + stage * kStageBytes;
          mbar_arrive_expect_tx(fb, kTxBytes);
          tma_load_2d(sst + kOffA, &tmA, fb, kb * 128, mt * 128);
          tma_load_2d(sst + kOffB, &tmB, fb, kb * 128, y_b);
          bulk_load(sst + kOffSfa, g.sfa + ((int64_t)mt * g.KB + kb) * kSfAtomBytes, kSfAtomBytes,
                    fb);
        }
        __syncwarp();
        issued_mask |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      buf ^= 1;
      stash_sfb(buf);
      e_cur = e_next;
      e_next = e_after;
    }
    // Drain: every copy this warp issued must have landed before the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        if (!(issued_mask & (1u << s))) continue;
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t par = (last_parity >> s) & 1u;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(fb, par) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf8_e4m3(128, kSingleN256 ? 256 : 128);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        if (!mbar_wait_bounded(smem_u32(&acce_bar), acc_phase ^ 1u, abort, g.status)) break;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < g.KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full_bar[stage]), phase, abort, g.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + stage * kStageBytes;
          const uint32_t sf = tmem + kColSf + stage * kSfSlotCols;
          tc_cp_sf_atom(sf, sdesc_sf_atom(st + kOffSfa));
          tc_cp_sf_atom(sf + 8, sdesc_sf_atom(st + kOffSfb));
          tc_cp_sf_atom(sf + 12, sdesc_sf_atom(st + kOffSfb + 512));
          const uint64_t ad = sdesc_k_sw128(st + kOffA);
          const uint64_t bd0 = sdesc_k_sw128(st + kOffB);
          const uint64_t bd1 = sdesc_k_sw128(st + kOffB + 16384);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
            // +32 bytes along K inside the 128-byte swizzle atom = +2 in the address field
            if constexpr (kSingleN256) {
              tc_mma_mxf8(tmem + 0, ad + 2 * k, bd0 + 2 * k, idesc, sf, sf + 8, acc);
            } else {
              tc_mma_mxf8(tmem + 0, ad + 2 * k, bd0 + 2 * k, idesc, sf, sf + 8, acc);
              tc_mma_mxf8(tmem + 128, ad + 2 * k, bd1 + 2 * k, idesc, sf, sf + 12, acc);
            }
          }
          tc_commit(smem_u32(&empty_bar[stage]));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&accf_bar));
        acc_phase ^= 1u;
      }
      // Drain: all MMAs / TMEM copies of this CTA complete before TMEM is freed.
      tc_commit(smem_u32(&drain_bar));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&drain_bar), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Eight warps, two per TMEM lane quadrant; thread = accumulator row, and
    // the two warps of a quadrant split the columns: FC2 -> columns
    // [128h, 128h+128); FC1 -> gate [64h, 64h+64) with the matching up
    // columns [128+64h, 192+64h), i.e. h columns [64h, 64h+64).
    // Phase 1 drains those 128 FP32 columns into BF16 pairs in registers (one
    // TMEM wait) and frees the accumulator at once, so the next tile's MMAs
    // overlap phase 2 (SwiGLU, quantisation, stores).  Every mode rounds the
    // accumulator to BF16 first: y and gate||up are stored as BF16, and the
    // fused SwiGLU reads gate/up after the same rounding as the unfused kernel.
    const int q = warp & 3;          // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;
    const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
    const int row_in_tile = q * 32 + lane;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const int mt = tile / g.NT, nt = tile - (tile / g.NT) * g.NT;
      if (!mbar_wait_bounded(smem_u32(&accf_bar), acc_phase, abort, g.status)) break;
      tc_fence_after();
      const int64_t row = (int64_t)mt * 128 + row_in_tile;
      // FC2: the second column half of a tile past H holds no output
      const bool active = !(MODE == kModeY && half == 1 && nt * 256 + 128 >= g.N);
      uint32_t pk[64];  // BF16 pairs of this warp's 128 accumulator columns
      if (active) {
        uint32_t r[4][32];
        if constexpr (MODE == kModeY) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tlane + half * 128 + c * 32, r[c]);
        } else {
          tmem_ld32(tlane + half * 64, r[0]);
          tmem_ld32(tlane + half * 64 + 32, r[1]);
          tmem_ld32(tlane + 128 + half * 64, r[2]);
          tmem_ld32(tlane + 128 + half * 64 + 32, r[3]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[c * 16 + j] =
                pack_bf16x2(__uint_as_float(r[c][2 * j]), __uint_as_float(r[c][2 * j + 1]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acce_bar));
      const uint32_t tile_par = acc_phase;  // alternates per tile
      acc_phase ^= 1u;

      if constexpr (MODE == kModeY) {
        if (active) {
          uint4* dst = reinterpret_cast<uint4*>(g.out + row * g.ld_out + (int64_t)nt * 256 + half * 128);
#pragma unroll
          for (int v = 0; v < 16; ++v)
            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if constexpr (MODE == kModeGU || MODE == kModeFusedGU) {
        uint16_t* base = g.out + row * g.ld_out + (int64_t)nt * 128 + half * 64;
        uint4* dg = reinterpret_cast<uint4*>(base);
        uint4* du = reinterpret_cast<uint4*>(base + g.inter);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          dg[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          du[v] = make_uint4(pk[32 + 4 * v], pk[32 + 4 * v + 1], pk[32 + 4 * v + 2], pk[32 + 4 * v + 3]);
        }
      }
      if constexpr (MODE == kModeFused || MODE == kModeFusedGU) {
        // gate pairs pk[0..31], up pairs pk[32..63] -> h[0..63]
        float h[64];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          h[2 * i] = swiglu(bf16_bits_to_float(pk[i] & 0xFFFFu), bf16_bits_to_float(pk[32 + i] & 0xFFFFu));
          h[2 * i + 1] = swiglu(bf16_bits_to_float(pk[i] >> 16), bf16_bits_to_float(pk[32 + i] >> 16));
          amax = fmaxf(amax, fmaxf(fabsf(h[2 * i]), fabsf(h[2 * i + 1])));
        }
        // row amax over both column halves (the two warps of this quadrant),
        // exchanged through shared memory, double-buffered by tile parity
        amax_sh[tile_par][half][row_in_tile] = amax;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&amax_bar[q]));
        if (!mbar_wait_bounded(smem_u32(&amax_bar[q]), tile_par, abort, g.status)) break;
        amax = fmaxf(amax, amax_sh[tile_par][half ^ 1][row_in_tile]);
        const int e = pow2_scale_exp(amax);
        const float inv = pow2_neg(e);
        uint4* dq = reinterpret_cast<uint4*>(g.hq + row * (int64_t)g.inter + (int64_t)nt * 128 + half * 64);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 16 * v + 4 * u;
            w[u] = e4m3x4(h[j] * inv, h[j + 1] * inv, h[j + 2] * inv, h[j + 3] * inv);
          }
          dq[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (half == 0)
          *reinterpret_cast<uint32_t*>(g.h_sf + sf_atom_offset(row, nt, g.IB)) =
              (uint32_t)(e + 127) * 0x01010101u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t gemm_set_attributes() {
  cudaError_t e;
  e = cudaFuncSetAttribute(fp8_grouped_gemm_kernel<kModeY>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fp8_grouped_gemm_kernel<kModeGU>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fp8_grouped_gemm_kernel<kModeFused>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fp8_grouped_gemm_kernel<kModeFusedGU>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
}

cudaError_t launch_gemm(GemmMode mode, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        const GemmArgs& g, int num_sms, cudaStream_t s) {
  const dim3 grid(num_sms), block(kThreads);
  switch (mode) {
    case kModeY:
      fp8_grouped_gemm_kernel<kModeY><<<grid, block, kDynSmem, s>>>(*tmA, *tmB, g);
      break;
    case kModeGU:
      fp8_grouped_gemm_kernel<kModeGU><<<grid, block, kDynSmem, s>>>(*tmA, *tmB, g);
      break;
    case kModeFused:
      fp8_grouped_gemm_kernel<kModeFused><<<grid, block, kDynSmem, s>>>(*tmA, *tmB, g);
      break;
    case kModeFusedGU:
      fp8_grouped_gemm_kernel<kModeFusedGU><<<grid, block, kDynSmem, s>>>(*tmA, *tmB, g);
      break;
  }
  return cudaGetLastError();
}

}  // namespace mm
