// gemm.cu -- steps 3 and 4 of the layer: the FC1 and FC2 grouped GEMMs over
// block-scaled FP8 expert weights (flashinfer PR #4069, Description: FC1 with
// fused SwiGLU + 1x128 quantization, then FC2; the DeepGEMM WGMMA kernels of
// that page are prior art for Hopper, not the design used here).
//
// GB300 design:
//  * tcgen05.mma kind::mxf8f6f4 with block scales: both operands E4M3, one
//    E8M0 scale per row per 32-wide K chunk.  Every scale of the layer is a
//    power of two, so 1x128 activation and 128x128 weight scales are applied
//    exactly by the tensor core while it accumulates in FP32 in tensor
//    memory: no per-K-block promotion through registers.  A scale atom holds
//    the bytes of four K blocks; the four MMAs of K block 4q + j select byte j
//    (the descriptor's scale-factor ids), so one tcgen05.cp per operand
//    serves four K blocks.  MXFP8 (GemmArgs::mx): the four bytes are the
//    scales of the four 32-wide chunks of one K block, so the atoms come
//    with every K block and MMA k selects byte k.
//  * Operands come from blocked buffers (every 128x128 block one contiguous
//    16 KB box: the weights from the bind step, A / hq from the quantisers),
//    one 3-D TMA box per block, 128-byte swizzle.
//  * Persistent CTAs walk a static tile list: 128 padded rows of one expert x
//    256 output columns, expert-major, so the m-tiles sharing a weight tile
//    run at the same time and hit it in L2.  The tile count and the m-tile ->
//    expert table come from device memory: no host synchronisation,
//    graph-capturable.
//  * Two variants (template PAIR):
//    - single CTA: one CTA per SM, M128 x N256 per MMA; a 4-stage ring of
//      50 KB stages (A 128x128 B, B two 128x128 B blocks, scale atoms).
//    - CTA pair (tcgen05 cta_group::2): two CTAs on the two SMs of a cluster
//      compute M256 x N256; each stages its own 128 A rows and one of the two
//      128-row B blocks (32 KB per K block instead of 48 KB), so a 6-stage
//      ring fits and more bytes are in flight per SM for the same MMA rate.
//      Both producers' TMA loads complete on the leader CTA's barrier, which
//      only the leader arms (with both CTAs' bytes); the leader issues the
//      scale copies and MMAs for the pair and multicasts its commits to both
//      CTAs; each CTA drains its own 128 accumulator rows.  Expert segments
//      are padded to 256 rows so a pair tile never straddles two experts.
//  * Warp roles (320 threads): warp 0 producer (TMA only: operand boxes, and
//    every fourth K block the A scale atom and the two B scale atoms built at
//    bind time), one thread of warp 1 issues the scale copies (tcgen05.cp)
//    and MMAs and probes the next stage while the current one computes,
//    warps 2-9 the epilogue (two per TMEM lane quadrant); the FOLD
//    instantiations add warps 10-11, the combine role (384 threads).
//  * Epilogues: FC2 -> BF16 y (TMA stores); FC1 unfused -> BF16 gate||up;
//    FC1 fused -> BF16-rounded gate/up, SwiGLU, 1x128 (or MXFP8 1x32)
//    re-quantisation to E4M3 + E8M0 atoms (bit-equal to the unfused path,
//    which runs the same device functions).
//  * kModeMega: FC1 then FC2 in one persistent launch.  Each fused FC1 tile
//    publishes its m-tile's count (fc1_done, release add after proxy-fenced
//    stores); an FC2 tile's producer waits for its m-tile's count before its
//    first TMA load of hq.  Every CTA takes its FC1 units before its FC2
//    units, so the waits always end (see the kernel's comment).
//  * Combine folded into FC2 (opt-in, single CTA; FOLD instantiations): the
//    FC2 epilogue counts each stored row into its token's per-n-tile count
//    and queues the pairs it completes for two extra warps, which combine
//    them (bit-identical to the combine kernel; slower than it on the
//    measured shapes).
//  * Launched as a programmatic dependent: the barrier / TMEM prologue
//    overlaps the previous kernel, the wait comes before the first global
//    read.
//  * Every wait is bounded (1 s); on expiry the kernel records
//    MOE_DEV_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"

namespace mm {

constexpr int kEpiWarps = 8;                   // two per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue
// Single-CTA launches that store y (FC2, or the megakernel) with the combine
// folded in are separate instantiations (FOLD) that carry two more warps:
// the combine role.  Every other launch compiles none of it.
constexpr int kCombineWarps = 2;
template <int MODE, bool PAIR, bool FOLD>
struct Roles {
  static constexpr bool kFold = FOLD && !PAIR && (MODE == kModeY || MODE == kModeMega);
  static constexpr int kThreads = mm::kThreads + (kFold ? 32 * kCombineWarps : 0);
};
constexpr int kCq = 256;  // the combine queue's slots (one per completed token n-tile)
constexpr uint32_t kTmemCols = 512;
// Scale factors live in TMEM after the accumulator (columns 0-255): four
// 16-column slots used in turn by successive groups of four K blocks (A atom
// at +0, B atoms at +8 and +12), so a copy never overwrites scales that MMAs
// of the previous three groups may still read.
constexpr uint32_t kColSf = 256, kSfSlotCols = 16;

template <bool PAIR>
struct StageCfg {
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr uint32_t kBRows = PAIR ? 128 : 256;       // B rows staged by this CTA
  static constexpr uint32_t kOffA = 0;                       // 128 rows x 128 B
  static constexpr uint32_t kOffB = 16384;                   // kBRows x 128 B
  static constexpr uint32_t kOffSfa = kOffB + kBRows * 128;  // one 512 B atom
  static constexpr uint32_t kOffSfb = kOffSfa + 512;         // two 512 B atoms
  static constexpr uint32_t kStageBytes = (kOffSfb + 1024 + 1023) / 1024 * 1024;
  static constexpr uint32_t kTxBytes = 16384 + kBRows * 128;  // operand bytes per CTA
  static constexpr uint32_t kTxAtomBytes = 3 * 512;            // + scale atoms, every 4th K block
  // FC2 output staging for TMA stores: 2 KB per epilogue warp, one 32-row x
  // 32-column BF16 box, 64-byte swizzle
  static constexpr bool kTmaStoreY = true;
  static constexpr uint32_t kOffYStage = (uint32_t)kStages * kStageBytes;
  static constexpr uint32_t kYStageBytes = kTmaStoreY ? 2048u * kEpiWarps : 0u;
  static constexpr size_t kDynSmem = (size_t)kStages * kStageBytes + kYStageBytes + 1024;
};

// Bounded wait until *count >= target (acquire at GPU scope), then a proxy
// fence so that the TMA loads this thread issues next observe what the
// threads that published the count wrote.
__device__ __noinline__ bool wait_count_geq(const int32_t* count, int target, volatile int* abort,
                                            uint32_t* status, uint64_t limit_ns) {
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

// The folded combine's arithmetic for up to NTOK (token, n-tile) pairs at
// once (one warp, eight columns per lane of the n-tile's 256; t < 0: none):
// out[t, c] = bf16_rn(fma chain over the active k = 0..K-1, ascending, of
// w[t, k] * y[inv_pad[t*K + k], c]) from +0 -- the combine kernel's
// arithmetic, so the output is bit-identical.  Every route row is loaded
// before any arithmetic, so the warp waits for one L2 round trip per call.
template <int NTOK>
__device__ __forceinline__ void fold_combine(const GemmArgs& gy, const int64_t (&t)[NTOK],
                                             const int (&nt)[NTOK], int lane) {
  const int K = gy.cmb_K;
  int c[NTOK];
  int p[NTOK][8];
  float wk[NTOK][8];
  uint4 v[NTOK][8];
#pragma unroll
  for (int j = 0; j < NTOK; ++j) {
    c[j] = nt[j] * 256 + lane * 8;
    const bool on = t[j] >= 0 && c[j] < gy.N;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      p[j][k] = (on && k < K) ? __ldg(gy.cmb_inv + t[j] * K + k) : -1;
      wk[j][k] = (on && k < K) ? __ldg(gy.cmb_w + t[j] * K + k) : 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < NTOK; ++j)
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[j][k] = p[j][k] >= 0
                    ? __ldcg(reinterpret_cast<const uint4*>(gy.out + (int64_t)p[j][k] * gy.ld_out + c[j]))
                    : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int j = 0; j < NTOK; ++j) {
    if (t[j] < 0 || c[j] >= gy.N) continue;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (p[j][k] < 0) continue;
      const uint32_t vv[4] = {v[j][k].x, v[j][k].y, v[j][k].z, v[j][k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(wk[j][k], bf16_bits_to_float(vv[i] & 0xFFFFu), acc[2 * i]);
        acc[2 * i + 1] = fmaf(wk[j][k], bf16_bits_to_float(vv[i] >> 16), acc[2 * i + 1]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(gy.cmb_out + t[j] * gy.N + c[j]) = o;
  }
}

// One launch runs the tiles of one GEMM (phase 0), or with MODE == kModeMega
// the FC1 tiles (phase 0: tmA/tmB/tmSfa/tmSfb, g) and then the FC2 tiles
// (phase 1: tmA2/tmB2/tmSfa2/tmSfb2, g2, tmY).  Units are numbered phase 0
// first.  A CTA pair takes every ustride-th unit in order.  A single CTA
// (g.sched set) takes unit blockIdx.x first and then the next unhanded one
// from a device counter (an atomic add), so CTAs that drew lighter units
// take more of them and the launch ends evenly; its producer passes each
// unit id to the MMA and epilogue roles through a small shared-memory ring.
// Either way units are handed out in increasing order, so every FC1 unit is
// taken by a running CTA before any FC2 unit, and FC2 tiles -- which wait
// for their m-tile's fc1_done count -- never hold up an FC1 tile: with every
// CTA resident the waits always end.
template <int MODE, bool PAIR, bool FOLD>
__global__ void __launch_bounds__(Roles<MODE, PAIR, FOLD>::kThreads, 1)
    fp8_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmSfa,
                            const __grid_constant__ CUtensorMap tmSfb,
                            const __grid_constant__ CUtensorMap tmY, const GemmArgs g,
                            const __grid_constant__ CUtensorMap tmA2,
                            const __grid_constant__ CUtensorMap tmB2,
                            const __grid_constant__ CUtensorMap tmSfa2,
                            const __grid_constant__ CUtensorMap tmSfb2, const GemmArgs g2) {
  using C = StageCfg<PAIR>;
  constexpr int kStages = C::kStages;
  constexpr bool kMega = MODE == kModeMega;
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar, acce_bar, drain_bar;
  __shared__ __align__(8) uint64_t amax_bar[4];  // per quadrant: both column halves posted
  __shared__ __align__(8) uint64_t fc1_bar[2];   // kModeMega: the epilogue warps' FC1 stores, by tile parity
  // the dynamic schedule's unit ring (single CTA): producer -> MMA + epilogue
  constexpr int kUnitSlots = 4;
  __shared__ int unit_ring[kUnitSlots];
  __shared__ __align__(8) uint64_t unit_full[kUnitSlots], unit_empty[kUnitSlots];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float amax_sh[2][2][128];  // [tile parity][column half][row] (fused epilogue)
  // the folded combine's queue: epilogue warps -> combine role, one entry per
  // completed (token, n-tile); an entry is published by writing its slot's
  // mark (index + 1)
  using R = Roles<MODE, PAIR, FOLD>;
  __shared__ int2 cq_item[R::kFold ? kCq : 1];
  __shared__ int cq_mark[R::kFold ? kCq : 1];
  __shared__ int cq_tail, cq_head, cq_freed, epi_done;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ustride = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const bool dyn = !PAIR && g.sched != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&accf_bar), 1);
    mbar_init(smem_u32(&acce_bar), kEpiWarps * (PAIR ? 2 : 1));
    mbar_init(smem_u32(&drain_bar), 1);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&amax_bar[i]), 2);
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&fc1_bar[i]), kEpiWarps);
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(smem_u32(&unit_full[i]), 1);
      mbar_init(smem_u32(&unit_empty[i]), 1 + kEpiWarps);  // the MMA thread + every epilogue warp
    }
    abort_sh = 0;
    if constexpr (R::kFold) {
      for (int i = 0; i < kCq; ++i) cq_mark[i] = 0;
      cq_tail = cq_head = cq_freed = epi_done = 0;
    }
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (PAIR) {
      prefetch_tensormap(&tmSfa);
      prefetch_tensormap(&tmSfb);
    }
    if (kMega) {
      prefetch_tensormap(&tmA2);
      prefetch_tensormap(&tmB2);
      if (PAIR) {
        prefetch_tensormap(&tmSfa2);
        prefetch_tensormap(&tmSfb2);
      }
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(&tmem_base_sh), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort = &abort_sh;
  // Everything above only touched this CTA's shared and tensor memory; the
  // routing tables and operands come from the previous kernels.
  pdl_wait();
  int mtiles = *g.total_mtiles;
  if (mtiles > g.max_mtiles) mtiles = g.max_mtiles;
  // work units: single CTA -> (m-tile, n-tile); pair -> (m-tile pair, n-tile)
  const int units_m = PAIR ? mtiles / 2 : mtiles;
  const int total0 = units_m * g.NT;
  const int total = total0 + (kMega ? units_m * g2.NT : 0);
  // unit u -> phase, m index (pair index for pairs), n-tile
  auto phase_of = [&](int u) { return (kMega && u >= total0) ? 1 : 0; };
  auto m_of = [&](int u, int ph) { return ph ? (u - total0) / g2.NT : u / g.NT; };
  auto nt_of = [&](int u, int ph, int m) { return ph ? (u - total0) - m * g2.NT : u - m * g.NT; };
  auto own_mtile = [&](int m) { return PAIR ? 2 * m + (int)rank : m; };
  // The folded combine's consumer (the combine role, and every epilogue warp
  // once its own tiles are done): lane 0 claims two queue entries and waits
  // (bounded) for each, or for the end -- every epilogue warp done and the
  // index past the tail; the warp combines the entries it found together.
  auto fold_consume = [&]() {
    const GemmArgs& gy = kMega ? g2 : g;
    while (true) {
      int r = 0;  // bit j: entry j found; -1: given up
      int2 it[2] = {make_int2(-1, 0), make_int2(-1, 0)};
      if (lane == 0) {
        const int base = atomicAdd(&cq_head, 2);
        for (int j = 0; j < 2 && r >= 0; ++j) {
          const int idx = base + j;
          const uint64_t t0 = globaltimer_ns();
          while (true) {
            if (*(volatile int*)&cq_mark[idx % kCq] == idx + 1) {
              __threadfence_block();
              it[j] = cq_item[idx % kCq];
              __threadfence_block();
              atomicAdd(&cq_freed, 1);
              r |= 1 << j;
              break;
            }
            if (*(volatile int*)&epi_done == kEpiWarps) {
              __threadfence_block();
              if (idx >= *(volatile int*)&cq_tail) break;
            }
            if (*abort) {
              r = -1;
              break;
            }
            if (globaltimer_ns() - t0 > g.wait_limit_ns) {
              *abort = 1;
              record_status(g.status, MOE_DEV_TIMEOUT);
              r = -1;
              break;
            }
            __nanosleep(64);
          }
        }
      }
      r = __shfl_sync(0xFFFFFFFFu, r, 0);
      if (r <= 0) break;
      const int64_t tt[2] = {(r & 1) ? (int64_t)__shfl_sync(0xFFFFFFFFu, it[0].x, 0) : -1,
                             (r & 2) ? (int64_t)__shfl_sync(0xFFFFFFFFu, it[1].x, 0) : -1};
      const int nn[2] = {__shfl_sync(0xFFFFFFFFu, it[0].y, 0), __shfl_sync(0xFFFFFFFFu, it[1].y, 0)};
      fold_combine<2>(gy, tt, nn, lane);
      if (!(r & 2)) break;  // the second index was past the end
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per unit the producer needs the expert id (a global table); it is
    // fetched one unit ahead so no dependent global load stalls the producer
    // at a tile boundary.  Every fourth K block the stage also carries the
    // scale atoms of the next four K blocks (A: this m-tile; B: the two
    // 128-row halves of the n-tile).  An FC2 tile of the megakernel first
    // waits until every FC1 tile of its m-tile has published its hq rows.
    auto expert_of = [&](int u) -> int {
      return u < total ? g.mtile_expert[(PAIR ? 2 : 1) * m_of(u, phase_of(u))] : 0;
    };
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued at least once, parity of last issue
    // the m-tile count an FC2 unit waits for, read (relaxed) one unit ahead
    auto count_of = [&](int u) -> int {
      return (kMega && u < total && phase_of(u))
                 ? ld_relaxed_gpu_s32(g2.fc1_done + own_mtile(m_of(u, 1)))
                 : 0;
    };
    // Dynamic schedule: the unit after the next is drawn (lane 0's atomic
    // add) at the start of each unit and read at its end, so the add's
    // latency overlaps the unit's loads; the unit ids go to the MMA and
    // epilogue roles through the ring (the last one, `total`, ends them).
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
    auto draw = [&]() -> int {  // lane 0 only
      return (int)gridDim.x + atomicAdd(g.sched, 1);
    };
    int u = unit0;
    int u_next = unit0 + ustride;
    if (dyn) {
      int v = 0;
      if (lane == 0 && u < total) v = draw();
      u_next = u < total ? __shfl_sync(0xFFFFFFFFu, v, 0) : total;
    }
    int e_next = expert_of(u);
    int count_next = count_of(u);
    for (; u < total && !*abort;) {
      if (dyn && !publish(u)) break;
      int pending = total;
      if (dyn && lane == 0 && u_next < total) pending = draw();
      const int ph = phase_of(u);
      const int m = m_of(u, ph);
      const int nt = nt_of(u, ph, m);
      const int mt = own_mtile(m);
      const int e = e_next;
      e_next = expert_of(u_next);
      const int count_seen = count_next;
      count_next = count_of(u_next);
      const int KB = ph ? g2.KB : g.KB, NB = ph ? g2.NB : g.NB, KQ = ph ? g2.KQ : g.KQ;
      const CUtensorMap* mA = ph ? &tmA2 : &tmA;
      const CUtensorMap* mB = ph ? &tmB2 : &tmB;
      const CUtensorMap* mSfa = ph ? &tmSfa2 : &tmSfa;
      const CUtensorMap* mSfb = ph ? &tmSfb2 : &tmSfb;
      const uint8_t* gsfa = ph ? g2.sfa : g.sfa;
      const uint8_t* gsfb = ph ? g2.sfb : g.sfb;
      if (kMega && ph == 1) {
        // usually complete by now (read a unit ago): the fence makes that
        // read an acquire; otherwise the bounded acquire-polling wait
        int ok = 1;
        if (lane == 0) {
          if (count_seen >= g2.fc1_ntiles) {
            fence_acq_rel_gpu();
            fence_proxy_async_global();
          } else {
            ok = wait_count_geq(g2.fc1_done + mt, g2.fc1_ntiles, abort, g.status, g.wait_limit_ns);
          }
        }
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      }
      // the n-tile's two 128-row weight blocks (the second clamped to the
      // first past N: those output columns are never stored); a pair CTA
      // stages the block of its rank
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
        if (g.watchdog_test && blockIdx.x == (PAIR ? 1u : 0u) && u == unit0 && kb == 2) {
          // watchdog test: this stage is never filled, so the MMA wait on it
          // expires; it is not counted as in flight for the drain below.  In
          // a pair the peer withholds its share: the leader still arms the
          // stage for both shares, so its full barrier never completes
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        if (lane == 0) {
          const uint32_t sst = sbase + stage * C::kStageBytes;
          // scale atoms: every fourth K block, or every K block under MXFP8
          const bool atoms = g.mx || (kb & 3) == 0;
          const int q = g.mx ? kb : kb >> 2;
          if constexpr (PAIR) {
            // Both CTAs' bytes complete on the leader's full barrier; only the
            // leader arrives (expecting both shares), so the peer's copies
            // may land before or after that arrival within the phase.
            const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
            if (leader)
              mbar_arrive_expect_tx(smem_u32(&full_bar[stage]),
                                    2 * (C::kTxBytes + (atoms ? C::kTxAtomBytes : 0u)));
            tma_load_3d_pair(sst + C::kOffA, mA, fb, 0, kb * 128, mt);
            tma_load_3d_pair(sst + C::kOffB, mB, fb, 0, kb * 128, rank ? wb1 : wb0);
            if (atoms) {
              tma_load_2d_pair(sst + C::kOffSfa, mSfa, fb, 0, (int)(sfa0 + q));
              tma_load_2d_pair(sst + C::kOffSfb, mSfb, fb, 0, (int)(sfb0 + q));
              tma_load_2d_pair(sst + C::kOffSfb + 512, mSfb, fb, 0, (int)(sfb1 + q));
            }
          } else {
            const uint32_t fb = smem_u32(&full_bar[stage]);
            mbar_arrive_expect_tx(fb, C::kTxBytes + (atoms ? C::kTxAtomBytes : 0u));
            tma_load_3d(sst + C::kOffA, mA, fb, 0, kb * 128, mt);
            tma_load_3d(sst + C::kOffB, mB, fb, 0, kb * 128, wb0);
            tma_load_3d(sst + C::kOffB + 16384, mB, fb, 0, kb * 128, wb1);
            if (atoms) {
              bulk_load(sst + C::kOffSfa, gsfa + (sfa0 + q) * kSfAtomBytes, kSfAtomBytes, fb);
              bulk_load(sst + C::kOffSfb, gsfb + (sfb0 + q) * kSfAtomBytes, kSfAtomBytes, fb);
              bulk_load(sst + C::kOffSfb + 512, gsfb + (sfb1 + q) * kSfAtomBytes, kSfAtomBytes, fb);
            }
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
    // Drain: every copy this CTA issued must have landed before the CTA exits
    // (the leader's full barriers also count the peer's bytes; the peer is
    // held by the cluster barrier at the end until the leader has drained).
    // After an abort the two producers may have stopped at different stages,
    // so the peer also gives its last copies a fixed 100 us to land.
    if (PAIR && !leader && lane == 0 && *abort) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 100000ull) {
      }
    }
    if (lane == 0 && leader) {
      for (int s = 0; s < kStages; ++s) {
        if (!(issued_mask & (1u << s))) continue;
        const uint32_t fb = smem_u32(&full_bar[s]);
        const uint32_t par = (last_parity >> s) & 1u;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(fb, par) && globaltimer_ns() - t0 < g.wait_limit_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      const uint32_t idesc0 = idesc_mxf8_e4m3(PAIR ? 256 : 128, 256);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      uint32_t group = 0;  // running count of scale-atom groups: TMEM slot = group % 4
      // Readiness of the next stage is probed right after the current
      // stage's MMAs are issued, so the probe's latency overlaps them; only a
      // stage found not ready goes through the (out-of-line) bounded wait.
      // The loop issues as few tcgen05 instructions as it can: the scale
      // atoms go to TMEM once per four K blocks.
      auto probe = [&](int s, uint32_t ph) {
        return PAIR ? mbar_test_wait_cluster(smem_u32(&full_bar[s]), ph)
                    : mbar_test_wait(smem_u32(&full_bar[s]), ph);
      };
      bool ready = probe(0, 0);
      uint32_t sf = tmem + kColSf;
      // the dynamic schedule's next unit, from the producer's ring
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
      for (int u = dyn ? take() : unit0; u < total; u = dyn ? take() : u + ustride) {
        if (!mbar_wait<PAIR>(smem_u32(&acce_bar), acc_phase ^ 1u, abort, g.status, g.wait_limit_ns)) break;
        tc_fence_after();
        bool ok = true;
        const int KB = phase_of(u) ? g2.KB : g.KB;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ready &&
              !mbar_wait_slow<PAIR>(smem_u32(&full_bar[stage]), phase, abort, g.status, g.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + stage * C::kStageBytes;
          const uint32_t j = (uint32_t)kb & 3u;
          if (g.mx || j == 0) {
            sf = tmem + kColSf + (group & 3u) * kSfSlotCols;
            ++group;
            if constexpr (PAIR) {
              tc_cp_sf_atom_pair(sf, sdesc_sf_atom(st + C::kOffSfa));
              tc_cp_sf_atom_pair(sf + 8, sdesc_sf_atom(st + C::kOffSfb));
              tc_cp_sf_atom_pair(sf + 12, sdesc_sf_atom(st + C::kOffSfb + 512));
            } else {
              tc_cp_sf_atom(sf, sdesc_sf_atom(st + C::kOffSfa));
              tc_cp_sf_atom(sf + 8, sdesc_sf_atom(st + C::kOffSfb));
              tc_cp_sf_atom(sf + 12, sdesc_sf_atom(st + C::kOffSfb + 512));
            }
          }
          const uint64_t ad = sdesc_k_sw128(st + C::kOffA);
          const uint64_t bd = sdesc_k_sw128(st + C::kOffB);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
            // scale byte of each TMEM scale word: K block j of the group, or
            // under MXFP8 the 32-wide chunk k of this K block
            const uint32_t sb = g.mx ? (uint32_t)k : j;
            const uint32_t idesc = idesc0 | (sb << 4) | (sb << 29);
            // +32 bytes along K inside the 128-byte swizzle atom = +2 in the address field
            if constexpr (PAIR)
              tc_mma_mxf8_pair(tmem, ad + 2 * k, bd + 2 * k, idesc, sf, sf + 8, acc);
            else
              tc_mma_mxf8(tmem, ad + 2 * k, bd + 2 * k, idesc, sf, sf + 8, acc);
          }
          const int done_stage = stage;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          ready = probe(stage, phase);
          if constexpr (PAIR)
            tc_commit_pair_multicast(smem_u32(&empty_bar[done_stage]), 0x3);
          else
            tc_commit(smem_u32(&empty_bar[done_stage]));
        }
        if (!ok) break;
        if constexpr (PAIR)
          tc_commit_pair_multicast(smem_u32(&accf_bar), 0x3);
        else
          tc_commit(smem_u32(&accf_bar));
        acc_phase ^= 1u;
      }
      // Drain: all MMAs / TMEM copies complete before TMEM is freed.
      if constexpr (PAIR)
        tc_commit_pair(smem_u32(&drain_bar));
      else
        tc_commit(smem_u32(&drain_bar));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(&drain_bar), 0) && globaltimer_ns() - t0 < g.wait_limit_ns) {
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
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
    // the accumulator-empty barrier lives in the leader CTA
    const uint32_t acce_addr = PAIR ? mapa_shared(smem_u32(&acce_bar), 0) : smem_u32(&acce_bar);
    uint32_t acc_phase = 0;
    uint32_t fc1_tiles = 0;  // kModeMega: FC1 tiles this CTA has published
    // the dynamic schedule's next unit: lane 0 takes it from the ring for the warp
    int slot = 0;
    uint32_t slot_ph = 0;
    // the folded combine: a lane queues a completed (token, n-tile) for the
    // combine role (bounded wait for a free slot)
    auto cq_push = [&](int tok, int ntile) -> bool {
      const int idx = atomicAdd(&cq_tail, 1);
      const uint64_t t0 = globaltimer_ns();
      while (idx - *(volatile int*)&cq_freed >= kCq) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > g.wait_limit_ns) {
          *abort = 1;
          record_status(g.status, MOE_DEV_TIMEOUT);
          return false;
        }
      }
      cq_item[idx % kCq] = make_int2(tok, ntile);
      __threadfence_block();
      *(volatile int*)&cq_mark[idx % kCq] = idx + 1;
      return true;
    };
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
    for (int u = dyn ? take() : unit0; u < total; u = dyn ? take() : u + ustride) {
      const int ph = phase_of(u);
      const int m = m_of(u, ph);
      const int nt = nt_of(u, ph, m);
      const int mt = own_mtile(m);
      // Routed rows of this m-tile, read before the accumulator wait (which
      // hides the loads).  The rest of the tile is its expert segment's
      // padding, which no later step reads: a warp whose 32 rows are all
      // padding skips the drain, the arithmetic and the stores.
      const int e_t = g.mtile_expert[mt];
      const bool live = q * 32 < g.pad_offsets[e_t] + g.counts[e_t] - mt * 128;
      // per-tensor format: the expert's factor on the FP32 accumulator (1
      // for the block-scaled formats, whose scales the tensor core applied)
      const float* pts = (kMega && ph) ? g2.pt_scale : g.pt_scale;
      const float acc_f = pts ? pts[e_t] : 1.0f;  // (unused without per-tensor scales)
      // the epilogue of this unit: the launch's mode, or per phase in the
      // megakernel (FC1 fused, with gate||up kept when its output is bound)
      const int em = kMega ? (ph ? kModeY : (g.out ? kModeFusedGU : kModeFused)) : MODE;
      const bool em_y = em == kModeY;
      const bool em_gu = em == kModeGU || em == kModeFusedGU;
      const bool em_fused = em == kModeFused || em == kModeFusedGU;
      // the folded combine: this row's token and its count target (two
      // column halves per active route), read before the accumulator wait
      int f_tok = -1, f_target = 0;
      if constexpr (R::kFold) {
        const GemmArgs& gy = (kMega && ph) ? g2 : g;
        if (em_y && gy.cmb_cnt && live) {
          const int64_t local = (int64_t)mt * 128 + row_in_tile - g.pad_offsets[e_t];
          if (local < g.counts[e_t]) {
            f_tok = gy.cmb_perm[gy.cmb_offsets[e_t] + local] / gy.cmb_K;
            int nact = 0;
            for (int k = 0; k < gy.cmb_K; ++k)
              nact += __ldg(gy.cmb_inv + (int64_t)f_tok * gy.cmb_K + k) >= 0;
            f_target = 2 * nact;
          }
        }
      }
      if (!mbar_wait(smem_u32(&accf_bar), acc_phase, abort, g.status, g.wait_limit_ns)) break;
      tc_fence_after();
      const int64_t row = (int64_t)mt * 128 + row_in_tile;
      // FC2: the second column half of a tile past H holds no output
      const bool active = live && !(em_y && half == 1 && nt * 256 + 128 >= (ph ? g2.N : g.N));
      uint32_t pk[64];  // BF16 pairs of this warp's 128 accumulator columns
      if (active) {
        uint32_t r[4][32];
        if (em_y) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tlane + half * 128 + c * 32, r[c]);
        } else {
          tmem_ld32(tlane + half * 64, r[0]);
          tmem_ld32(tlane + half * 64 + 32, r[1]);
          tmem_ld32(tlane + 128 + half * 64, r[2]);
          tmem_ld32(tlane + 128 + half * 64 + 32, r[3]);
        }
        tmem_ld_wait();
        if (pts) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[c * 16 + j] = pack_bf16x2(__fmul_rn(__uint_as_float(r[c][2 * j]), acc_f),
                                           __fmul_rn(__uint_as_float(r[c][2 * j + 1]), acc_f));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[c * 16 + j] =
                  pack_bf16x2(__uint_as_float(r[c][2 * j]), __uint_as_float(r[c][2 * j + 1]));
        }
      }
      // The TMEM reads above have completed (tcgen05.wait::ld); the arrive
      // passes no data through memory, so in the pair it is relaxed: a
      // cluster-scope release would first wait for this thread's
      // outstanding global stores of the previous tile.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)
          mbar_arrive_cluster_relaxed(acce_addr);
        else
          mbar_arrive(acce_addr);
      }
      const uint32_t tile_par = acc_phase;  // alternates per tile
      acc_phase ^= 1u;

      // Stores are 32 bytes per thread per instruction (whole sectors): every
      // destination below is 32-byte aligned (row pitches and tile offsets are
      // multiples of 64 bytes, buffers 1024-byte aligned).
      if (em_y && C::kTmaStoreY) {
        // TMA stores: the warp's 32 rows x 128 columns leave in four 32x32
        // boxes through its 2 KB staging buffer; row r's 16-byte chunk j sits
        // at r*64 + ((j ^ ((r >> 1) & 3)) * 16) (the 64-byte swizzle).
        if (active) {
          const uint32_t buf = sbase + C::kOffYStage + (uint32_t)(warp - 2) * 2048u;
          uint8_t* bufp = smem + C::kOffYStage + (warp - 2) * 2048;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (lane == 0) bulk_wait_group_read0();  // previous box has left the buffer
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int pj = j ^ ((lane >> 1) & 3);
              *reinterpret_cast<uint4*>(bufp + lane * 64 + pj * 16) =
                  make_uint4(pk[c * 16 + 4 * j], pk[c * 16 + 4 * j + 1], pk[c * 16 + 4 * j + 2],
                             pk[c * 16 + 4 * j + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmY, buf, nt * 256 + half * 128 + c * 32, mt * 128 + q * 32);
              bulk_commit_group();
            }
          }
        }
      } else if (em_y) {
        if (active) {
          uint16_t* dst = g.out + row * g.ld_out + (int64_t)nt * 256 + half * 128;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            st_global_v8(dst + 16 * v, pk[8 * v], pk[8 * v + 1], pk[8 * v + 2], pk[8 * v + 3],
                         pk[8 * v + 4], pk[8 * v + 5], pk[8 * v + 6], pk[8 * v + 7]);
        }
      }
      if constexpr (R::kFold) {
        // The combine folded in: once this warp's y boxes are written (not
        // only read out of shared memory) and made visible at GPU scope,
        // each routed row adds one to its token's count for the n-tile (a
        // tile half past H stores nothing and counts all the same).  The
        // lane whose add completes a count queues the (token, n-tile) for
        // the combine role.
        const GemmArgs& gy = (kMega && ph) ? g2 : g;
        if (em_y && gy.cmb_cnt && live) {
          if (lane == 0 && active) {
            bulk_wait_group0();
            fence_proxy_async_global();
          }
          __syncwarp();
          __threadfence();
          const bool done =
              f_tok >= 0 && atomicAdd(gy.cmb_cnt + (int64_t)f_tok * gy.NT + nt, 1) == f_target - 1;
          if (__any_sync(0xFFFFFFFFu, done)) __threadfence();
          const int ok = done ? (cq_push(f_tok, nt) ? 1 : 0) : 1;
          if (!__all_sync(0xFFFFFFFFu, ok)) break;
        }
      }
      if (em_gu && active) {
        uint16_t* dg = g.out + row * g.ld_out + (int64_t)nt * 128 + half * 64;
        uint16_t* du = dg + g.inter;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          st_global_v8(dg + 16 * v, pk[8 * v], pk[8 * v + 1], pk[8 * v + 2], pk[8 * v + 3],
                       pk[8 * v + 4], pk[8 * v + 5], pk[8 * v + 6], pk[8 * v + 7]);
          st_global_v8(du + 16 * v, pk[32 + 8 * v], pk[32 + 8 * v + 1], pk[32 + 8 * v + 2],
                       pk[32 + 8 * v + 3], pk[32 + 8 * v + 4], pk[32 + 8 * v + 5],
                       pk[32 + 8 * v + 6], pk[32 + 8 * v + 7]);
        }
      }
      if (em_fused && g.pt_rh && active) {
        // per-tensor: h * (1 / h_scale) rounded once in float, then E4M3;
        // the block scale is 1 (no amax exchange)
        float h[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          h[2 * i] = swiglu(bf16_bits_to_float(pk[i] & 0xFFFFu),
                            bf16_bits_to_float(pk[32 + i] & 0xFFFFu));
          h[2 * i + 1] = swiglu(bf16_bits_to_float(pk[i] >> 16), bf16_bits_to_float(pk[32 + i] >> 16));
        }
        const float rh = *g.pt_rh;
        uint8_t* dq = g.hq + blocked_offset(row, (int64_t)nt * 128 + half * 64, g.inter);
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          uint32_t w[8];
#pragma unroll
          for (int uu = 0; uu < 8; ++uu) {
            const int j = 32 * v + 4 * uu;
            w[uu] = e4m3x4(__fmul_rn(h[j], rh), __fmul_rn(h[j + 1], rh), __fmul_rn(h[j + 2], rh),
                           __fmul_rn(h[j + 3], rh));
          }
          st_global_v8(dq + 32 * v, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
        }
        if (half == 0) g.h_sf[sf_atom_offset(row, nt, g.IB)] = (uint8_t)127;
      } else if (em_fused && g.mx && active) {
        // MXFP8: this thread's 64 h columns are two whole 32-wide chunks of
        // its row, so each gets its scale without any exchange
        float h[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          h[2 * i] = swiglu(bf16_bits_to_float(pk[i] & 0xFFFFu),
                            bf16_bits_to_float(pk[32 + i] & 0xFFFFu));
          h[2 * i + 1] = swiglu(bf16_bits_to_float(pk[i] >> 16), bf16_bits_to_float(pk[32 + i] >> 16));
        }
        uint8_t* dq = g.hq + blocked_offset(row, (int64_t)nt * 128 + half * 64, g.inter);
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[32 * v + i]));
          const int e = pow2_scale_exp(amax);
          const float inv = pow2_neg(e);
          uint32_t w[8];
#pragma unroll
          for (int uu = 0; uu < 8; ++uu) {
            const int jx = 32 * v + 4 * uu;
            w[uu] = e4m3x4(h[jx] * inv, h[jx + 1] * inv, h[jx + 2] * inv, h[jx + 3] * inv);
          }
          st_global_v8(dq + 32 * v, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
          g.h_sf[sf_atom_offset(row, 4 * nt + 2 * half + v, 4 * g.IB)] = (uint8_t)(e + 127);
        }
      } else if (em_fused && !g.mx && !g.pt_rh && !active) {
        // a padding quadrant (both of its warps decide alike) still completes
        // this tile's phase of the amax exchange, which every 1x128 fused
        // tile advances once (MXFP8 tiles have no exchange)
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&amax_bar[q]));
        if (!mbar_wait(smem_u32(&amax_bar[q]), tile_par, abort, g.status, g.wait_limit_ns)) break;
      } else if (em_fused && !g.mx && !g.pt_rh) {
        // gate pairs pk[0..31], up pairs pk[32..63] -> h[0..63]
        float h[64];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          h[2 * i] = swiglu(bf16_bits_to_float(pk[i] & 0xFFFFu),
                            bf16_bits_to_float(pk[32 + i] & 0xFFFFu));
          h[2 * i + 1] = swiglu(bf16_bits_to_float(pk[i] >> 16), bf16_bits_to_float(pk[32 + i] >> 16));
          amax = fmaxf(amax, fmaxf(fabsf(h[2 * i]), fabsf(h[2 * i + 1])));
        }
        // row amax over both column halves (the two warps of this quadrant),
        // exchanged through shared memory, double-buffered by tile parity
        amax_sh[tile_par][half][row_in_tile] = amax;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&amax_bar[q]));
        if (!mbar_wait(smem_u32(&amax_bar[q]), tile_par, abort, g.status, g.wait_limit_ns)) break;
        amax = fmaxf(amax, amax_sh[tile_par][half ^ 1][row_in_tile]);
        const int e = pow2_scale_exp(amax);
        const float inv = pow2_neg(e);
        uint8_t* dq = g.hq + blocked_offset(row, (int64_t)nt * 128 + half * 64, g.inter);
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          uint32_t w[8];
#pragma unroll
          for (int uu = 0; uu < 8; ++uu) {
            const int j = 32 * v + 4 * uu;
            w[uu] = e4m3x4(h[j] * inv, h[j + 1] * inv, h[j + 2] * inv, h[j + 3] * inv);
          }
          st_global_v8(dq + 32 * v, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
        }
        if (half == 0) g.h_sf[sf_atom_offset(row, nt, g.IB)] = (uint8_t)(e + 127);
      }
      if (kMega && ph == 0) {
        // Publish this FC1 tile: every epilogue warp's hq / scale stores are
        // ordered before its arrival (proxy fence: FC2 reads them by TMA);
        // one thread waits for all eight arrivals, then adds to the m-tile's
        // count with release semantics.  Two barriers alternate by tile, so a
        // warp already on the next FC1 tile cannot arrive on this phase.
        fence_proxy_async_global();
        __syncwarp();
        const uint32_t fb = smem_u32(&fc1_bar[fc1_tiles & 1u]);
        if (lane == 0) mbar_arrive(fb);
        if (warp == 2) {
          int ok = 1;
          if (lane == 0) {
            ok = mbar_wait(fb, (fc1_tiles >> 1) & 1u, abort, g.status, g.wait_limit_ns) ? 1 : 0;
            if (ok) {
              __threadfence();
              red_release_gpu_add(g.fc1_done + mt, 1);
            }
          }
          if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;  // the whole warp leaves together
        }
        ++fc1_tiles;
      }
    }
    if constexpr (R::kFold) {
      // nothing more to queue from this warp; it helps combine what is left
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        atomicAdd(&epi_done, 1);
      }
      if ((kMega ? g2 : g).cmb_cnt) fold_consume();
    }
  } else if constexpr (R::kFold) {
    // ------------------------------------------------------------ combine role
    // With the combine folded in (the FC2 args carry cmb_cnt), two warps
    // combine the (token, n-tile) pairs whose counts the epilogue completed:
    // a count is complete at 2 x the token's active routes (both column
    // halves of every route row stored), and the lane whose add completes it
    // queues the pair.  Tokens with no active route get +0 rows here, as the
    // combine kernel gives them.
    const GemmArgs& gy = kMega ? g2 : g;
    if (gy.cmb_cnt) {
      const int cw = warp - 2 - kEpiWarps;
      const int K = gy.cmb_K;
      const int64_t zstride = (int64_t)gridDim.x * kCombineWarps * 32;
      for (int64_t t = ((int64_t)blockIdx.x * kCombineWarps + cw) * 32 + lane; t < gy.cmb_T;
           t += zstride) {
        int nact = 0;
        for (int k = 0; k < K; ++k) nact += __ldg(gy.cmb_inv + t * K + k) >= 0;
        if (nact == 0)
          for (int c = 0; c < gy.N; c += 8)
            *reinterpret_cast<uint4*>(gy.cmb_out + t * gy.N + c) = make_uint4(0u, 0u, 0u, 0u);
      }
      fold_consume();
    }
  }

  if constexpr ((MODE == kModeY || MODE == kModeMega) && StageCfg<PAIR>::kTmaStoreY) {
    // this warp's output boxes are written
    if (warp >= 2 && warp < 2 + kEpiWarps && lane == 0) bulk_wait_group0();
  }
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if constexpr (PAIR) cluster_sync_all();  // neither CTA frees TMEM the pair still uses
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE, bool PAIR, bool FOLD = false>
static cudaError_t set_attr() {
  return cudaFuncSetAttribute(fp8_grouped_gemm_kernel<MODE, PAIR, FOLD>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)StageCfg<PAIR>::kDynSmem);
}

cudaError_t gemm_set_attributes() {
  cudaError_t e;
  if ((e = set_attr<kModeY, false>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeGU, false>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeFused, false>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeFusedGU, false>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeY, true>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeGU, true>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeFused, true>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeFusedGU, true>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeMega, false>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeY, false, true>()) != cudaSuccess) return e;
  if ((e = set_attr<kModeMega, false, true>()) != cudaSuccess) return e;
  return set_attr<kModeMega, true>();
}

static cudaLaunchAttribute pair_cluster_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = 2;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  return a;
}

// Largest number of CTA pairs that can be resident at once (0 if none).
int gemm_max_pairs() {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr = pair_cluster_attr();
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = StageCfg<true>::kDynSmem;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fp8_grouped_gemm_kernel<kModeY, true, false>, &cfg) !=
      cudaSuccess)
    return 0;
  return n;
}

// Single-phase launches pass the phase-0 maps and args again as phase 1
// (unused).  The single-CTA kernel reads scale atoms by bulk copy, so its
// atom maps are placeholders too.
template <int MODE>
static cudaError_t launch_mode(bool pair, const CUtensorMap* tmA, const CUtensorMap* tmB,
                               const CUtensorMap* tmSfa, const CUtensorMap* tmSfb,
                               const CUtensorMap* tmA2, const CUtensorMap* tmB2,
                               const CUtensorMap* tmSfa2, const CUtensorMap* tmSfb2,
                               const CUtensorMap* tmY, const GemmArgs& g, const GemmArgs& g2,
                               int ctas, cudaStream_t s, bool pdl) {
  // the combine folded into FC2 (single CTAs): the FC2 args carry its counters
  const bool fold = !pair && (MODE == kModeY || MODE == kModeMega) &&
                    (MODE == kModeMega ? g2.cmb_cnt : g.cmb_cnt) != nullptr;
  if (fold) {
    constexpr int M = (MODE == kModeY || MODE == kModeMega) ? MODE : kModeY;  // (others never fold)
    return launch_k(fp8_grouped_gemm_kernel<M, false, true>, dim3(ctas),
                    dim3(Roles<M, false, true>::kThreads), StageCfg<false>::kDynSmem, s, pdl, nullptr,
                    *tmA, *tmB, *tmA, *tmA, *tmY, g, *tmA2, *tmB2, *tmA2, *tmA2, g2);
  }
  if (!pair)
    return launch_k(fp8_grouped_gemm_kernel<MODE, false, false>, dim3(ctas),
                    dim3(Roles<MODE, false, false>::kThreads), StageCfg<false>::kDynSmem, s, pdl,
                    nullptr, *tmA, *tmB, *tmA, *tmA, *tmY, g, *tmA2, *tmB2, *tmA2, *tmA2, g2);
  const cudaLaunchAttribute cluster = pair_cluster_attr();
  return launch_k(fp8_grouped_gemm_kernel<MODE, true, false>, dim3(ctas), dim3(Roles<MODE, true, false>::kThreads),
                  StageCfg<true>::kDynSmem, s, pdl, &cluster, *tmA, *tmB, *tmSfa, *tmSfb, *tmY, g,
                  *tmA2, *tmB2, *tmSfa2, *tmSfb2, g2);
}

cudaError_t launch_gemm(GemmMode mode, bool pair, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        const CUtensorMap* tmSfa, const CUtensorMap* tmSfb, const CUtensorMap* tmY,
                        const GemmArgs& g, int ctas, cudaStream_t s, bool pdl) {
#define MM_ONE_PHASE(M) \
  launch_mode<M>(pair, tmA, tmB, tmSfa, tmSfb, tmA, tmB, tmSfa, tmSfb, tmY, g, g, ctas, s, pdl)
  switch (mode) {
    case kModeY: return MM_ONE_PHASE(kModeY);
    case kModeGU: return MM_ONE_PHASE(kModeGU);
    case kModeFused: return MM_ONE_PHASE(kModeFused);
    case kModeFusedGU: return MM_ONE_PHASE(kModeFusedGU);
    case kModeMega: break;  // two phases: launch_gemm_mega
  }
#undef MM_ONE_PHASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_mega(bool pair, const CUtensorMap* tmA, const CUtensorMap* tmB,
                             const CUtensorMap* tmSfa, const CUtensorMap* tmSfb,
                             const CUtensorMap* tmA2, const CUtensorMap* tmB2,
                             const CUtensorMap* tmSfa2, const CUtensorMap* tmSfb2,
                             const CUtensorMap* tmY, const GemmArgs& g, const GemmArgs& g2, int ctas,
                             cudaStream_t s, bool pdl) {
  if (!g2.fc1_done || g2.fc1_ntiles != g.NT) return cudaErrorInvalidValue;
  return launch_mode<kModeMega>(pair, tmA, tmB, tmSfa, tmSfb, tmA2, tmB2, tmSfa2, tmSfb2, tmY, g,
                                g2, ctas, s, pdl);
}

}  // namespace mm
