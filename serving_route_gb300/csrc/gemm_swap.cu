// gemm_swap.cu -- the token-as-N ("swap-AB") form of the FC1 / FC2 grouped
// GEMMs for small forwards (flashinfer PR #4069, Limitations: the fused FC1
// epilogue had no small-M swap-AB variant; flashinfer PR #4688: token-bucket
// heuristics that pick swap-AB token tiles for small token counts).
//
// When no expert receives more than NTOK routed rows (NTOK in {16, 32, 64};
// certain when num_tokens <= NTOK, because a token routes to an expert at
// most once), each unit of the single-CTA kernel -- one 128-row m-tile of an
// expert times 256 weight rows -- is computed transposed: the weight rows are
// the M = 128 operand of two MMAs per K step (FC1: the gate block and the up
// block of one 128-wide slice of I; FC2: two 128-row blocks of W2), and the
// first NTOK rows of the m-tile are the N operand.  A stage holds 32 KB of
// weights and NTOK x 128 B of activations -- instead of 32 KB of weights and
// 16 KB of activation rows that are mostly segment padding -- so 6 stages
// (NTOK = 16) or 5 fit, with more weight bytes in flight per SM; and the two
// NTOK-column accumulators are double-buffered in tensor memory, so the MMAs
// of the next unit start while the epilogue drains this one.
//
// The epilogue sees the accumulator transposed: TMEM lane = weight row (an h
// index, or an output column), TMEM column = token.  FC1: gate and up of h
// index i for token t sit in the same lane, SwiGLU is elementwise, and the
// 1x128 requantisation of token t reduces over the 128 lanes (a warp max,
// then the four lane quadrants through shared memory; MXFP8's 32-wide chunks
// are one warp's lanes).  FC2: y[t, c] as BF16, 64 contiguous bytes per warp
// and token.  The arithmetic is the M128 x N256 kernel's (gate and up rounded
// to BF16 before SwiGLU, the same swiglu() and encoders), checked against the
// oracle; the fused epilogue is bit-equal to this kernel's unfused path.
// Every wait is bounded (1 s) and a timed-out CTA winds down as the other
// GEMM kernel's do.
#include "common.cuh"
#include "internal.h"

namespace mm {
namespace {

constexpr int kSwEpiWarps = 8;                    // two per TMEM lane quadrant
constexpr int kSwThreads = 64 + 32 * kSwEpiWarps;  // producer, MMA, epilogue
constexpr uint32_t kSwSlotCols = 16;              // scale slot: W0 atom +0, W1 atom +4, X atom +8

template <int NTOK>
struct SwapCfg {
  static constexpr int kStages = NTOK == 16 ? 6 : 5;
  static constexpr uint32_t kOffW0 = 0;                     // 128 weight rows x 128 B
  static constexpr uint32_t kOffW1 = 16384;                 // the second 128 weight rows
  static constexpr uint32_t kOffX = 32768;                  // NTOK activation rows x 128 B
  static constexpr uint32_t kOffSfW0 = kOffX + NTOK * 128;  // 512 B scale atoms
  static constexpr uint32_t kOffSfW1 = kOffSfW0 + 512;
  static constexpr uint32_t kOffSfX = kOffSfW1 + 512;
  static constexpr uint32_t kStageBytes = (kOffSfX + 512 + 1023) / 1024 * 1024;
  static constexpr uint32_t kTxBytes = 32768 + NTOK * 128;
  static constexpr uint32_t kTxAtomBytes = 3 * 512;
  static constexpr size_t kDynSmem = (size_t)kStages * kStageBytes + 1024;
  // tensor memory: accumulator buffer b at 2*NTOK*b ([D0 | D1], NTOK columns
  // each), then four scale slots
  static constexpr uint32_t kColSf = 4 * NTOK;
  static constexpr uint32_t kTmemCols =
      kColSf + 4 * kSwSlotCols <= 128 ? 128 : (kColSf + 4 * kSwSlotCols <= 256 ? 256 : 512);
};

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]);

template <>
__device__ __forceinline__ void tmem_ld_cols<8>(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld_cols<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ uint8_t e4m3x1(float v) { return (uint8_t)(e4m3x2(v, 0.f) & 0xFFu); }

// The combine of one token's 256 output columns [c0, c0 + 256) by one warp
// (8 columns per lane): out[t, c] = bf16_rn(fma chain over the active k =
// 0..K-1, ascending, of w[t, k] * y[inv_pad[t*K + k], c]) from +0 -- the
// combine kernel's arithmetic, so the output is bit-identical.  The K route
// rows are loaded together, from L2 (other warps and CTAs stored them).
__device__ __forceinline__ void combine_token(const GemmArgs& gy, const uint16_t* y, int64_t ld,
                                              int64_t t, int c0, int N, int lane) {
  const int c = c0 + lane * 8;
  if (c >= N) return;
  const int K = gy.cmb_K;
  int p[8];
  float wk[8];
  uint4 v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    p[k] = k < K ? __ldg(gy.cmb_inv + t * K + k) : -1;
    wk[k] = k < K ? __ldg(gy.cmb_w + t * K + k) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k)
    v[k] = p[k] >= 0 ? __ldcg(reinterpret_cast<const uint4*>(y + (int64_t)p[k] * ld + c))
                     : make_uint4(0u, 0u, 0u, 0u);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
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
  *reinterpret_cast<uint4*>(gy.cmb_out + t * N + c) = o;
}

// Bounded wait until *count >= target (acquire), then a proxy fence for the
// TMA loads that follow (as in the M128 x N256 kernel).
__device__ __noinline__ bool swap_wait_count_geq(const int32_t* count, int target,
                                                 volatile int* abort, uint32_t* status,
                                                 uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu_s32(count) < target) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      record_status(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
  fence_proxy_async_global();
  return true;
}

// One launch runs the units of one GEMM (phase 0), or with MODE == kModeMega
// the FC1 units and then the FC2 units (phase 1: tmX2 / tmW2, g2).  Units are
// those of the M128 x N256 kernel (m-tile x 256 weight rows, expert-major),
// taken in the same static or counter order, so the fc1_done waits of the
// one-launch form end for the same reason.
template <int MODE, int NTOK>
__global__ void __launch_bounds__(kSwThreads, 1)
    fp8_swap_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmW, const GemmArgs g,
                         const __grid_constant__ CUtensorMap tmX2,
                         const __grid_constant__ CUtensorMap tmW2, const GemmArgs g2) {
  using C = SwapCfg<NTOK>;
  constexpr int kStages = C::kStages;
  constexpr bool kMega = MODE == kModeMega;
  constexpr int NT2 = NTOK / 2;  // token columns per epilogue warp
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2], drain_bar;
  __shared__ __align__(8) uint64_t fc1_bar[2];
  __shared__ __align__(8) uint64_t amax_bar[2];  // per token half: its four quadrant warps posted
  constexpr int kUnitSlots = 4;
  __shared__ int unit_ring[kUnitSlots];
  __shared__ __align__(8) uint64_t unit_full[kUnitSlots], unit_empty[kUnitSlots];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float amax_sh[2][2][4][NT2];  // [tile parity][token half][lane quadrant][token]

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit0 = (int)blockIdx.x;
  const int ustride = (int)gridDim.x;
  const bool dyn = g.sched != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accf_bar[b]), 1);
      mbar_init(smem_u32(&acce_bar[b]), kSwEpiWarps);
      mbar_init(smem_u32(&fc1_bar[b]), kSwEpiWarps);
      mbar_init(smem_u32(&amax_bar[b]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(smem_u32(&unit_full[i]), 1);
      mbar_init(smem_u32(&unit_empty[i]), 1 + kSwEpiWarps);
    }
    abort_sh = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
    if (kMega) {
      prefetch_tensormap(&tmX2);
      prefetch_tensormap(&tmW2);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort = &abort_sh;
  pdl_wait();
  int mtiles = *g.total_mtiles;
  if (mtiles > g.max_mtiles) mtiles = g.max_mtiles;
  const int total0 = mtiles * g.NT;
  const int total = total0 + (kMega ? mtiles * g2.NT : 0);
  auto phase_of = [&](int u) { return (kMega && u >= total0) ? 1 : 0; };
  auto m_of = [&](int u, int ph) { return ph ? (u - total0) / g2.NT : u / g.NT; };
  auto nt_of = [&](int u, int ph, int m) { return ph ? (u - total0) - m * g2.NT : u - m * g.NT; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    auto expert_of = [&](int u) -> int { return u < total ? g.mtile_expert[m_of(u, phase_of(u))] : 0; };
    auto count_of = [&](int u) -> int {
      return (kMega && u < total && phase_of(u)) ? ld_relaxed_gpu_s32(g2.fc1_done + m_of(u, 1)) : 0;
    };
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, last_parity = 0;
    int slot = 0;
    uint32_t slot_ph = 0;
    auto publish = [&](int v) -> bool {
      if (!mbar_wait(smem_u32(&unit_empty[slot]), slot_ph ^ 1u, abort, g.status, g.wait_limit_ns))
        return false;
      if (lane == 0) {
        unit_ring[slot] = v;
        mbar_arrive(smem_u32(&unit_full[slot]));
      }
      __syncwarp();
      if (++slot == kUnitSlots) {
        slot = 0;
        slot_ph ^= 1u;
      }
      return true;
    };
    int u = unit0;
    int u_next = unit0 + ustride;
    if (dyn) {
      int v = 0;
      if (lane == 0 && u < total) v = (int)gridDim.x + atomicAdd(g.sched, 1);
      u_next = u < total ? __shfl_sync(0xFFFFFFFFu, v, 0) : total;
    }
    int e_next = expert_of(u);
    int count_next = count_of(u);
    while (u < total && !*abort) {
      if (dyn && !publish(u)) break;
      int pending = total;
      if (dyn && lane == 0 && u_next < total) pending = (int)gridDim.x + atomicAdd(g.sched, 1);
      const int ph = phase_of(u);
      const int mt = m_of(u, ph);
      const int nt = nt_of(u, ph, mt);
      const int e = e_next;
      e_next = expert_of(u_next);
      const int count_seen = count_next;
      count_next = count_of(u_next);
      const int KB = ph ? g2.KB : g.KB, NB = ph ? g2.NB : g.NB, KQ = ph ? g2.KQ : g.KQ;
      const CUtensorMap* mX = ph ? &tmX2 : &tmX;
      const CUtensorMap* mW = ph ? &tmW2 : &tmW;
      const uint8_t* gsfa = ph ? g2.sfa : g.sfa;
      const uint8_t* gsfb = ph ? g2.sfb : g.sfb;
      if (kMega && ph == 1) {
        int okw = 1;
        if (lane == 0) {
          if (count_seen >= g2.fc1_ntiles) {
            fence_acq_rel_gpu();
            fence_proxy_async_global();
          } else {
            okw = swap_wait_count_geq(g2.fc1_done + mt, g2.fc1_ntiles, abort, g.status,
                                      g.wait_limit_ns);
          }
        }
        if (!__shfl_sync(0xFFFFFFFFu, okw, 0)) break;
      }
      // the unit's two 128-row weight blocks (the second clamped to the first
      // past N: those outputs are never stored)
      const int nb0 = 2 * nt, nb1 = (2 * nt + 1 < NB) ? 2 * nt + 1 : 2 * nt;
      const int wb0 = e * NB + nb0, wb1 = e * NB + nb1;
      const int64_t sfb0 = ((int64_t)e * NB + nb0) * KQ, sfb1 = ((int64_t)e * NB + nb1) * KQ;
      const int64_t sfa0 = (int64_t)mt * KQ;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort, g.status, g.wait_limit_ns)) {
          ok = false;
          break;
        }
        if (g.watchdog_test && blockIdx.x == 0u && u == unit0 && kb == 2) {
          // watchdog test: this stage is never filled, so the MMA wait on it expires
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        if (lane == 0) {
          const uint32_t sst = sbase + stage * C::kStageBytes;
          const bool atoms = g.mx || (kb & 3) == 0;
          const int q = g.mx ? kb : kb >> 2;
          const uint32_t fb = smem_u32(&full_bar[stage]);
          mbar_arrive_expect_tx(fb, C::kTxBytes + (atoms ? C::kTxAtomBytes : 0u));
          tma_load_3d(sst + C::kOffW0, mW, fb, 0, kb * 128, wb0);
          tma_load_3d(sst + C::kOffW1, mW, fb, 0, kb * 128, wb1);
          tma_load_3d(sst + C::kOffX, mX, fb, 0, kb * 128, mt);
          if (atoms) {
            bulk_load(sst + C::kOffSfW0, gsfb + (sfb0 + q) * kSfAtomBytes, kSfAtomBytes, fb);
            bulk_load(sst + C::kOffSfW1, gsfb + (sfb1 + q) * kSfAtomBytes, kSfAtomBytes, fb);
            bulk_load(sst + C::kOffSfX, gsfa + (sfa0 + q) * kSfAtomBytes, kSfAtomBytes, fb);
          }
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
      const int drawn = __shfl_sync(0xFFFFFFFFu, pending, 0);
      u = u_next;
      u_next = dyn ? drawn : u + ustride;
    }
    if (dyn && !*abort) publish(total);  // ends the MMA and epilogue roles
    // Drain: every copy this CTA issued must have landed before it exits.
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        if (!(issued_mask & (1u << s))) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&full_bar[s]), (last_parity >> s) & 1u) &&
               globaltimer_ns() - t0 < g.wait_limit_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc0 = idesc_mxf8_e4m3(128, NTOK);
      int stage = 0;
      uint32_t phase = 0, uses[2] = {0u, 0u};
      uint32_t group = 0;
      bool ready = mbar_test_wait(smem_u32(&full_bar[0]), 0);
      uint32_t sf = tmem + C::kColSf;
      int slot = 0;
      uint32_t slot_ph = 0;
      auto take = [&]() -> int {
        if (!mbar_wait(smem_u32(&unit_full[slot]), slot_ph, abort, g.status, g.wait_limit_ns))
          return total;
        const int v = unit_ring[slot];
        mbar_arrive(smem_u32(&unit_empty[slot]));
        if (++slot == kUnitSlots) {
          slot = 0;
          slot_ph ^= 1u;
        }
        return v;
      };
      int i = 0;
      for (int u = dyn ? take() : unit0; u < total; u = dyn ? take() : u + ustride, ++i) {
        const int b = i & 1;
        if (!mbar_wait(smem_u32(&acce_bar[b]), (uses[b] & 1u) ^ 1u, abort, g.status, g.wait_limit_ns))
          break;
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)(2 * NTOK * b), d1 = d0 + NTOK;
        bool ok = true;
        const int KB = phase_of(u) ? g2.KB : g.KB;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ready && !mbar_wait_slow<false>(smem_u32(&full_bar[stage]), phase, abort, g.status,
                                               g.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + stage * C::kStageBytes;
          const uint32_t j = (uint32_t)kb & 3u;
          if (g.mx || j == 0) {
            sf = tmem + C::kColSf + (group & 3u) * kSwSlotCols;
            ++group;
            tc_cp_sf_atom(sf, sdesc_sf_atom(st + C::kOffSfW0));
            tc_cp_sf_atom(sf + 4, sdesc_sf_atom(st + C::kOffSfW1));
            tc_cp_sf_atom(sf + 8, sdesc_sf_atom(st + C::kOffSfX));
          }
          const uint64_t w0 = sdesc_k_sw128(st + C::kOffW0);
          const uint64_t w1 = sdesc_k_sw128(st + C::kOffW1);
          const uint64_t xd = sdesc_k_sw128(st + C::kOffX);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
            const uint32_t sbyte = g.mx ? (uint32_t)k : j;
            const uint32_t idesc = idesc0 | (sbyte << 4) | (sbyte << 29);
            tc_mma_mxf8(d0, w0 + 2 * k, xd + 2 * k, idesc, sf, sf + 8, acc);
            tc_mma_mxf8(d1, w1 + 2 * k, xd + 2 * k, idesc, sf + 4, sf + 8, acc);
          }
          const int done_stage = stage;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          ready = mbar_test_wait(smem_u32(&full_bar[stage]), phase);
          tc_commit(smem_u32(&empty_bar[done_stage]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&accf_bar[b]));
        ++uses[b];
      }
      tc_commit(smem_u32(&drain_bar));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&drain_bar), 0) && globaltimer_ns() - t0 < g.wait_limit_ns) {
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Two warps per TMEM lane quadrant: lane = weight row i = 32q + lane of
    // the unit's 128-row blocks; the two warps of a quadrant take the token
    // columns [NT2*half, NT2*half + NT2).
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int irow = q * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
    const int col0 = half * NT2;
    uint32_t uses[2] = {0u, 0u};
    uint32_t fc1_tiles = 0;
    int slot = 0;
    uint32_t slot_ph = 0;
    auto take = [&]() -> int {
      int v = total;
      if (lane == 0 &&
          mbar_wait(smem_u32(&unit_full[slot]), slot_ph, abort, g.status, g.wait_limit_ns)) {
        v = unit_ring[slot];
        mbar_arrive(smem_u32(&unit_empty[slot]));
      }
      if (++slot == kUnitSlots) {
        slot = 0;
        slot_ph ^= 1u;
      }
      return __shfl_sync(0xFFFFFFFFu, v, 0);
    };
    // With the combine folded into FC2, a token whose routes are all masked
    // completes no count: one warp writes its output row, +0 (as the combine
    // kernel does), before any unit (the routing is complete here).
    const GemmArgs& gc = kMega ? g2 : g;
    if (gc.cmb_cnt && blockIdx.x == 0 && warp == 2) {
      const int N = gc.N;
      for (int t0 = 0; t0 < gc.cmb_T; t0 += 32) {
        const int t = t0 + lane;
        bool dead = false;
        if (t < gc.cmb_T) {
          int nact = 0;
          for (int k = 0; k < gc.cmb_K; ++k) nact += __ldg(gc.cmb_inv + (int64_t)t * gc.cmb_K + k) >= 0;
          dead = nact == 0;
        }
        uint32_t m = __ballot_sync(0xFFFFFFFFu, dead);
        while (m) {
          const int src = __ffs(m) - 1;
          m &= m - 1;
          for (int c = lane * 8; c < N; c += 256)
            *reinterpret_cast<uint4*>(gc.cmb_out + (int64_t)(t0 + src) * N + c) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    int i = 0;
    for (int u = dyn ? take() : unit0; u < total; u = dyn ? take() : u + ustride, ++i) {
      const int b = i & 1;
      const int ph = phase_of(u);
      const int mt = m_of(u, ph);
      const int nt = nt_of(u, ph, mt);
      const int e_t = g.mtile_expert[mt];
      int live = g.pad_offsets[e_t] + g.counts[e_t] - mt * 128;  // routed rows of this m-tile
      live = live < 0 ? 0 : (live > NTOK ? NTOK : live);
      const float* pts = (kMega && ph) ? g2.pt_scale : g.pt_scale;
      const float acc_f = pts ? pts[e_t] : 1.0f;
      const int em = kMega ? (ph ? kModeY : (g.out ? kModeFusedGU : kModeFused)) : MODE;
      const bool em_y = em == kModeY;
      const bool em_gu = em == kModeGU || em == kModeFusedGU;
      const bool em_fused = em == kModeFused || em == kModeFusedGU;
      if (!mbar_wait(smem_u32(&accf_bar[b]), uses[b] & 1u, abort, g.status, g.wait_limit_ns)) break;
      ++uses[b];
      tc_fence_after();
      uint32_t r0[NT2], r1[NT2];
      tmem_ld_cols<NT2>(tlane + (uint32_t)(2 * NTOK * b + col0), r0);
      tmem_ld_cols<NT2>(tlane + (uint32_t)(2 * NTOK * b + NTOK + col0), r1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acce_bar[b]));
      float a0[NT2], a1[NT2];
#pragma unroll
      for (int c = 0; c < NT2; ++c) {
        a0[c] = pts ? __fmul_rn(__uint_as_float(r0[c]), acc_f) : __uint_as_float(r0[c]);
        a1[c] = pts ? __fmul_rn(__uint_as_float(r1[c]), acc_f) : __uint_as_float(r1[c]);
      }
      const int64_t row0 = (int64_t)mt * 128 + col0;  // GEMM row of this warp's first token
      if (em_y) {
        // y[row, 256nt + i] from D0, y[row, 256nt + 128 + i] from D1 (when inside H)
        const int N = ph ? g2.N : g.N;
        const bool second = nt * 256 + 128 < N;
        uint16_t* out = ph ? g2.out : g.out;
        const int64_t ld = ph ? g2.ld_out : g.ld_out;
#pragma unroll
        for (int c = 0; c < NT2; ++c) {
          if (col0 + c >= live) break;
          uint16_t* dst = out + (row0 + c) * ld + (int64_t)nt * 256 + irow;
          dst[0] = (uint16_t)(pack_bf16x2(a0[c], 0.f) & 0xFFFFu);
          if (second) dst[128] = (uint16_t)(pack_bf16x2(a1[c], 0.f) & 0xFFFFu);
        }
        const GemmArgs& gy = (kMega && ph) ? g2 : g;
        if (gy.cmb_cnt) {
          // The combine, folded in.  Each token's 256 columns of this unit
          // are stored by the four lane-quadrant warps of its token half;
          // every warp counts each of its live tokens once its y stores are
          // visible (each lane's fence, then the warp's sync), into the
          // token's count for this n-tile.  The warp whose add completes a
          // token's count (4 x its active routes) combines that token's
          // columns of the n-tile.
          __threadfence();
          __syncwarp();
          int64_t tok = -1;
          bool complete = false;
          if (lane < NT2 && col0 + lane < live) {
            const int64_t pos = row0 + lane - g.pad_offsets[e_t] + gy.cmb_offsets[e_t];
            tok = gy.cmb_perm[pos] / gy.cmb_K;
            int nact = 0;
            for (int k = 0; k < gy.cmb_K; ++k) nact += __ldg(gy.cmb_inv + tok * gy.cmb_K + k) >= 0;
            const int old = atomicAdd(gy.cmb_cnt + tok * gy.NT + nt, 1);
            complete = old == 4 * nact - 1;
          }
          uint32_t todo = __ballot_sync(0xFFFFFFFFu, complete);
          if (todo) __threadfence();
          while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int64_t t = __shfl_sync(0xFFFFFFFFu, tok, src);
            combine_token(gy, out, ld, t, nt * 256, N, lane);
          }
        }
      }
      if (em_gu) {
        // gate column 128nt + i from D0, up column I + 128nt + i from D1
#pragma unroll
        for (int c = 0; c < NT2; ++c) {
          if (col0 + c >= live) break;
          uint16_t* dst = g.out + (row0 + c) * g.ld_out + (int64_t)nt * 128 + irow;
          dst[0] = (uint16_t)(pack_bf16x2(a0[c], 0.f) & 0xFFFFu);
          dst[g.inter] = (uint16_t)(pack_bf16x2(a1[c], 0.f) & 0xFFFFu);
        }
      }
      if (em_fused) {
        float h[NT2];
#pragma unroll
        for (int c = 0; c < NT2; ++c) h[c] = swiglu(bf16_round(a0[c]), bf16_round(a1[c]));
        if (g.pt_rh) {
          // per-tensor: h * (1 / h_scale), block scale 1
          const float rh = *g.pt_rh;
#pragma unroll
          for (int c = 0; c < NT2; ++c) {
            if (col0 + c >= live) break;
            g.hq[blocked_offset(row0 + c, (int64_t)nt * 128 + irow, g.inter)] = e4m3x1(__fmul_rn(h[c], rh));
            if (irow == 0) g.h_sf[sf_atom_offset(row0 + c, nt, g.IB)] = (uint8_t)127;
          }
        } else if (g.mx) {
          // MXFP8: this warp's 32 lanes are one 32-wide chunk of h
#pragma unroll
          for (int c = 0; c < NT2; ++c) {
            const int e = pow2_scale_exp(warp_max(fabsf(h[c])));
            if (col0 + c >= live) continue;
            g.hq[blocked_offset(row0 + c, (int64_t)nt * 128 + irow, g.inter)] = e4m3x1(h[c] * pow2_neg(e));
            if (lane == 0) g.h_sf[sf_atom_offset(row0 + c, 4 * nt + q, 4 * g.IB)] = (uint8_t)(e + 127);
          }
        } else {
          // 1x128: the row amax over the 128 lanes -- a warp max per token,
          // then the four quadrant warps of this token half through shared
          // memory, double-buffered by tile parity, behind a bounded
          // mbarrier that every fused tile advances once
          const uint32_t par = fc1_tiles & 1u;
#pragma unroll
          for (int c = 0; c < NT2; ++c) {
            const float m = warp_max(fabsf(h[c]));
            if (lane == c) amax_sh[par][half][q][c] = m;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&amax_bar[half]));
          if (!mbar_wait(smem_u32(&amax_bar[half]), par, abort, g.status, g.wait_limit_ns)) break;
#pragma unroll
          for (int c = 0; c < NT2; ++c) {
            const float m = fmaxf(fmaxf(amax_sh[par][half][0][c], amax_sh[par][half][1][c]),
                                  fmaxf(amax_sh[par][half][2][c], amax_sh[par][half][3][c]));
            const int e = pow2_scale_exp(m);
            if (col0 + c >= live) continue;
            g.hq[blocked_offset(row0 + c, (int64_t)nt * 128 + irow, g.inter)] = e4m3x1(h[c] * pow2_neg(e));
            if (irow == 0) g.h_sf[sf_atom_offset(row0 + c, nt, g.IB)] = (uint8_t)(e + 127);
          }
        }
      }
      if (em_fused || em_gu) ++fc1_tiles;  // tile parity of the amax exchange
      if (kMega && ph == 0) {
        // publish this FC1 unit for the FC2 units of its m-tile (as in the
        // M128 x N256 kernel; two barriers alternate by published tile)
        const uint32_t pub = fc1_tiles - 1u;
        fence_proxy_async_global();
        __syncwarp();
        const uint32_t fb = smem_u32(&fc1_bar[pub & 1u]);
        if (lane == 0) mbar_arrive(fb);
        if (warp == 2) {
          int okp = 1;
          if (lane == 0) {
            okp = mbar_wait(fb, (pub >> 1) & 1u, abort, g.status, g.wait_limit_ns) ? 1 : 0;
            if (okp) {
              __threadfence();
              red_release_gpu_add(g.fc1_done + mt, 1);
            }
          }
          if (!__shfl_sync(0xFFFFFFFFu, okp, 0)) break;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int MODE, int NTOK>
cudaError_t swap_attr() {
  return cudaFuncSetAttribute(fp8_swap_gemm_kernel<MODE, NTOK>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)SwapCfg<NTOK>::kDynSmem);
}

template <int NTOK>
cudaError_t swap_attrs() {
  cudaError_t e;
  if ((e = swap_attr<kModeY, NTOK>()) != cudaSuccess) return e;
  if ((e = swap_attr<kModeGU, NTOK>()) != cudaSuccess) return e;
  if ((e = swap_attr<kModeFused, NTOK>()) != cudaSuccess) return e;
  if ((e = swap_attr<kModeFusedGU, NTOK>()) != cudaSuccess) return e;
  return swap_attr<kModeMega, NTOK>();
}

template <int NTOK>
cudaError_t launch_swap_n(GemmMode mode, const CUtensorMap* tmX, const CUtensorMap* tmW,
                          const CUtensorMap* tmX2, const CUtensorMap* tmW2, const GemmArgs& g,
                          const GemmArgs& g2, int ctas, cudaStream_t s, bool pdl) {
  const size_t smem = SwapCfg<NTOK>::kDynSmem;
#define MM_SWAP(M)                                                                            \
  launch_k(fp8_swap_gemm_kernel<M, NTOK>, dim3(ctas), dim3(kSwThreads), smem, s, pdl, nullptr, \
           *tmX, *tmW, g, *tmX2, *tmW2, g2)
  switch (mode) {
    case kModeY: return MM_SWAP(kModeY);
    case kModeGU: return MM_SWAP(kModeGU);
    case kModeFused: return MM_SWAP(kModeFused);
    case kModeFusedGU: return MM_SWAP(kModeFusedGU);
    case kModeMega: return MM_SWAP(kModeMega);
  }
#undef MM_SWAP
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t gemm_swap_set_attributes() {
  cudaError_t e;
  if ((e = swap_attrs<16>()) != cudaSuccess) return e;
  if ((e = swap_attrs<32>()) != cudaSuccess) return e;
  return swap_attrs<64>();
}

cudaError_t launch_gemm_swap(GemmMode mode, int ntok, const CUtensorMap* tmX, const CUtensorMap* tmW,
                             const CUtensorMap* tmX2, const CUtensorMap* tmW2, const GemmArgs& g,
                             const GemmArgs& g2, int ctas, cudaStream_t s, bool pdl) {
  if (mode == kModeMega && (!g2.fc1_done || g2.fc1_ntiles != g.NT)) return cudaErrorInvalidValue;
  switch (ntok) {
    case 16: return launch_swap_n<16>(mode, tmX, tmW, tmX2, tmW2, g, g2, ctas, s, pdl);
    case 32: return launch_swap_n<32>(mode, tmX, tmW, tmX2, tmW2, g, g2, ctas, s, pdl);
    case 64: return launch_swap_n<64>(mode, tmX, tmW, tmX2, tmW2, g, g2, ctas, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mm
