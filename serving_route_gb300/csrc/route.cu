// route.cu -- step 1 of the layer: route validation, expert histogram,
// device-side exclusive scan and stable scatter of the routes into
// per-expert contiguous segments ("compact" in the forward diagram of
// flashinfer PR #4069; validation rules of flashinfer PR #6398 "fuse Rubin
// MegaMoE forward preparation": expert-id bounds, no duplicate routes, finite
// scores on active routes, masked slots (-1) may carry any score).
//
// By default one cooperative kernel (route_fused, below) when its blocks can
// all be resident; otherwise -- and under an SM budget, and for the
// no-allocation entry point -- three small kernels, no host synchronisation
// (the second and third are launched as programmatic dependents, so their
// launch overlaps the previous kernel):
//   route_count   per 128-token block: validate, per-block expert histogram
//   route_scan    one CTA: expert totals, unpadded and padded (128 or 256
//                 rows per GEMM segment) exclusive scans, per-block bases,
//                 the 128-row m-tile -> expert table
//   route_scatter per 128-token block: stable rank of every route inside its
//                 expert (flat route id order, via warp match + per-warp
//                 prefix), writing perm / inv / inv_pad
// Route ids outside [-1, E) are flagged and then treated as masked, so no
// later kernel indexes out of bounds whatever the input.
#include "common.cuh"
#include "internal.h"

namespace mm {

constexpr int kRouteTokens = 128;  // tokens per block (one per thread in route_count)

__global__ void __launch_bounds__(kRouteTokens) route_count_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, int T, int K, int E, int check,
    int32_t* __restrict__ block_counts, uint32_t* __restrict__ status) {
  pdl_trigger();  // the scan may launch now; it waits for this grid to complete
  extern __shared__ int32_t hist[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int t = blockIdx.x * kRouteTokens + threadIdx.x;
  uint32_t err = 0;
  if (t < T) {
    int ids[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) ids[k] = (k < K) ? idx[(int64_t)t * K + k] : -1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k >= K) break;
      const int id = ids[k];
      if (id == -1) continue;
      if (id < 0 || id >= E) {
        err |= MOE_DEV_ROUTE_RANGE;
        continue;
      }
      atomicAdd(&hist[id], 1);
      if (check) {
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2)
          if (k2 < k && ids[k2] == id) err |= MOE_DEV_ROUTE_DUP;
        const float wv = w[(int64_t)t * K + k];
        if (!isfinite(wv)) err |= MOE_DEV_ROUTE_NONFINITE;
      }
    }
  }
  if (err) record_status(status, err);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    block_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// Exclusive scan of one value per thread across the CTA (blockDim.x <= 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = (blockDim.x + 31) >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = (lane < nwarps) ? warp_sums[lane] : 0;
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xFFFFFFFFu, si, o);
      if (lane >= o) si += n;
    }
    if (lane < nwarps) warp_sums[lane] = si - s;
    if (lane == nwarps - 1) *total = si;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) route_scan_kernel(
    const int32_t* __restrict__ block_counts, int nb, int E, int pad_rows, int64_t rows_alloc,
    int max_mtiles,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ pad_offsets,
    int32_t* __restrict__ base_u, int32_t* __restrict__ base_p, int32_t* __restrict__ mtile_expert,
    int32_t* __restrict__ total_mtiles, uint32_t* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  __shared__ int warp_sums[32];
  __shared__ int tot_u, tot_p;
  const int e = threadIdx.x;
  int c = 0;
  if (e < E)
    for (int b = 0; b < nb; ++b) c += block_counts[(int64_t)b * E + e];
  const int cp = (c + pad_rows - 1) / pad_rows * pad_rows;  // GEMM segment of the expert
  const int off_u = block_exclusive_scan(c, warp_sums, &tot_u);
  const int off_p = block_exclusive_scan(cp, warp_sums, &tot_p);
  if (e < E) {
    counts[e] = c;
    offsets[e] = off_u;
    pad_offsets[e] = off_p;
    int run = 0;
    for (int b = 0; b < nb; ++b) {
      base_u[(int64_t)b * E + e] = off_u + run;
      base_p[(int64_t)b * E + e] = off_p + run;
      run += block_counts[(int64_t)b * E + e];
    }
    const int m0 = off_p >> 7, m1 = (off_p + cp) >> 7;
    for (int m = m0; m < m1 && m < max_mtiles; ++m) mtile_expert[m] = e;
  }
  if (e == 0) {
    offsets[E] = tot_u;
    pad_offsets[E] = tot_p;
    if ((int64_t)tot_p > rows_alloc) {
      record_status(status, MOE_DEV_CAPACITY);
      *total_mtiles = 0;
    } else {
      *total_mtiles = tot_p >> 7;
    }
  }
}

__global__ void __launch_bounds__(kRouteTokens) route_scatter_kernel(
    const int32_t* __restrict__ idx, int T, int K, int E, int64_t rows_alloc,
    const int32_t* __restrict__ base_u, const int32_t* __restrict__ base_p,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int32_t* __restrict__ inv_pad) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t wh[];  // [4 warps][E]: per-warp counts, then running bases
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kRouteTokens / 32;
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();
  // routes of this warp: tokens [t0, t0 + 32), flat ids [r0, r1)
  const int64_t t0 = (int64_t)blockIdx.x * kRouteTokens + warp * 32;
  const int64_t r0 = t0 * K;
  const int64_t r1 = min((int64_t)T, t0 + 32) * K;
  for (int64_t r = r0 + lane; r < r1; r += 32) {
    const int id = idx[r];
    if (id >= 0 && id < E) atomicAdd(&wh[warp * E + id], 1);
  }
  __syncthreads();
  // exclusive prefix over the warps of the block, per expert
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = wh[w * E + e];
      wh[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  int32_t* my = wh + warp * E;
  const int32_t* bu = base_u + (int64_t)blockIdx.x * E;
  const int32_t* bp = base_p + (int64_t)blockIdx.x * E;
  // the warp's route ids, loaded together (at most K <= 8 rounds of 32)
  int idv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t r = r0 + j * 32 + lane;
    idv[j] = r < r1 ? idx[r] : -1;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t rb = r0 + j * 32;
    if (rb >= r1) break;  // the same for the whole warp
    const int64_t r = rb + lane;
    const bool in = r < r1;
    const int id = idv[j];
    const bool act = in && id >= 0 && id < E;
    const unsigned amask = __ballot_sync(0xFFFFFFFFu, act);
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, act ? id : -1) & amask;
    int rank = 0, base = 0;
    if (act) {
      rank = __popc(peers & ((1u << lane) - 1u));
      base = my[id];
    }
    __syncwarp();
    if (act) {
      const int local = base + rank;
      const int pos = bu[id] + local;
      const int64_t ppos = (int64_t)bp[id] + local;
      perm[pos] = (int32_t)r;
      inv[r] = pos;
      inv_pad[r] = (ppos < rows_alloc) ? (int32_t)ppos : -1;
      // the highest lane of each peer group advances that expert's running base
      if ((peers >> lane) == 1u) my[id] = base + __popc(peers);
    } else if (in) {
      inv[r] = -1;
      inv_pad[r] = -1;
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// One-kernel routing: the three steps above in one cooperative launch, with a
// grid-wide barrier where the kernel boundaries were.  The outputs are the
// same bit for bit: the same per-warp counting, scans and rank rule.
//   phase 1  validate this block's tokens and count their routes per warp
//            and expert; publish the block's histogram row
//   barrier  every block arrives on a counter zeroed before the forward; the
//            launch is cooperative (all blocks resident), and the wait is
//            bounded all the same
//   phase 2  every block reads the whole [nb][E] histogram (eight loads in
//            flight per thread, summed with shared-memory atomics): expert
//            totals, its own prefix over earlier blocks, the unpadded and
//            padded exclusive scans; the expert-level outputs (counts,
//            offsets, m-tile table) are spread over the blocks
//   phase 3  the stable scatter of route_scatter, bases from shared memory
// ---------------------------------------------------------------------------
// 512 tokens per block (a warp per 32 tokens, as in route_scatter): four
// times fewer histogram rows than the 128-token blocks of the three-kernel
// form, and four times the threads to read them after the barrier.
constexpr int kFusedTokens = 512;
constexpr int kRouteWarps = kFusedTokens / 32;

inline size_t route_fused_smem(int E) { return sizeof(int32_t) * (size_t)(kRouteWarps + 2) * E; }

__global__ void __launch_bounds__(kFusedTokens) route_fused_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, int T, int K, int E, int check,
    int pad_rows, int64_t rows_alloc, int max_mtiles, int32_t* __restrict__ block_counts,
    uint32_t* __restrict__ grid_sync, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ pad_offsets, int32_t* __restrict__ mtile_expert,
    int32_t* __restrict__ total_mtiles, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
    int32_t* __restrict__ inv_pad, uint32_t* __restrict__ status, uint64_t wait_limit_ns,
    int withhold, uint32_t* __restrict__ zero_base, int zero_words) {
  extern __shared__ int32_t sm[];
  int32_t* wh = sm;                   // [warps][E]: per-warp counts, then running bases
  int32_t* bu = sm + kRouteWarps * E;  // [E]: expert totals, then this block's unpadded bases
  int32_t* bp = bu + E;               // [E]: this block's prefix, then its padded bases
  __shared__ int warp_sums[32];
  __shared__ int tot_u, tot_p, passed;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = (int)gridDim.x, b = (int)blockIdx.x;
  // a one-block routing is the forward's first kernel and its only block:
  // it clears the forward's status word and counters itself (the barrier
  // below orders the clearing before this block's first status update)
  if (nb == 1)
    for (int i = tid; i < zero_words; i += blockDim.x) zero_base[i] = 0u;
  for (int i = tid; i < kRouteWarps * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();

  // ---- phase 1
  const int t = b * kFusedTokens + tid;
  uint32_t err = 0;
  if (t < T) {
    int ids[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) ids[k] = (k < K) ? idx[(int64_t)t * K + k] : -1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k >= K) break;
      const int id = ids[k];
      if (id == -1) continue;
      if (id < 0 || id >= E) {
        err |= MOE_DEV_ROUTE_RANGE;
        continue;
      }
      atomicAdd(&wh[warp * E + id], 1);
      if (check) {
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2)
          if (k2 < k && ids[k2] == id) err |= MOE_DEV_ROUTE_DUP;
        const float wv = w[(int64_t)t * K + k];
        if (!isfinite(wv)) err |= MOE_DEV_ROUTE_NONFINITE;
      }
    }
  }
  if (err) record_status(status, err);
  __syncthreads();
  // One block (at most 512 tokens): its histogram is the whole one, so the
  // expert totals go straight to shared memory (no earlier block: prefix 0)
  // and the grid barrier and the histogram's round trip through global
  // memory are skipped.
  const bool one = nb == 1;
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int v = 0; v < kRouteWarps; ++v) c += wh[v * E + e];
    block_counts[(int64_t)b * E + e] = c;
    if (one) {
      bu[e] = c;
      bp[e] = 0;
    }
  }

  // The flat route ids of this warp's phase-3 routes (tokens [t0, t0 + 32),
  // at most K <= 8 rounds of 32), loaded now so that their latency overlaps
  // the barrier; idx is an input of the forward, no kernel writes it.
  const int64_t t0 = (int64_t)b * kFusedTokens + warp * 32;
  const int64_t r0 = t0 * K;
  const int64_t r1 = min((int64_t)T, t0 + 32) * K;
  int idv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t r = r0 + j * 32 + lane;
    idv[j] = r < r1 ? idx[r] : -1;
  }

  // ---- grid barrier
  __syncthreads();
  if (one) {
    if (tid == 0) passed = 1;
  } else if (tid == 0) {
    __threadfence();  // this block's histogram row before its arrival
    if (b != withhold) atomicAdd(grid_sync, 1u);  // withhold: the barrier test's missing block
    bool ok = true;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu_u32(grid_sync) < (uint32_t)nb) {
      if (globaltimer_ns() - t0 > wait_limit_ns) {
        ok = false;
        break;
      }
    }
    if (!ok) record_status(status, MOE_DEV_TIMEOUT);
    __threadfence();
    passed = ok ? 1 : 0;
  }
  __syncthreads();
  pdl_trigger();  // quant_dispatch may launch; it waits for this grid to complete
  if (!passed) {
    // No routing this forward (the status says why): this block's routes are
    // marked unrouted, so every later kernel skips them; total_mtiles keeps
    // the 0 written before the forward unless block 0 got through.
    const int64_t q0 = (int64_t)b * kFusedTokens * K;
    const int64_t q1 = min((int64_t)T, (int64_t)(b + 1) * kFusedTokens) * K;
    for (int64_t r = q0 + tid; r < q1; r += blockDim.x) {
      inv[r] = -1;
      inv_pad[r] = -1;
    }
    return;
  }

  // ---- phase 2
  // expert totals and this block's prefix over the earlier blocks: the
  // (block, expert) entries spread over the threads, eight loads in flight
  // per thread, summed with shared-memory atomics
  if (!one) {
    for (int e = tid; e < E; e += blockDim.x) {
      bu[e] = 0;
      bp[e] = 0;
    }
  }
  __syncthreads();
  const int n_ent = one ? 0 : nb * E;
  for (int p0 = tid; p0 < n_ent; p0 += 8 * kFusedTokens) {
    int c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = p0 + j * kFusedTokens;
      c[j] = p < n_ent ? __ldcg(block_counts + p) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int p = p0 + j * kFusedTokens;
      if (c[j] != 0) {
        const int v = p / E, e = p - v * E;
        atomicAdd(&bu[e], c[j]);
        if (v < b) atomicAdd(&bp[e], c[j]);
      }
    }
  }
  __syncthreads();
  // thread tid scans the run of experts [e0, e1)
  const int per = (E + kFusedTokens - 1) / kFusedTokens;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int su = 0, sp = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = bu[e];
    su += c;
    sp += (c + pad_rows - 1) / pad_rows * pad_rows;
  }
  int run_u = block_exclusive_scan(su, warp_sums, &tot_u);
  int run_p = block_exclusive_scan(sp, warp_sums, &tot_p);
  for (int e = e0; e < e1; ++e) {
    const int c = bu[e], cp = (c + pad_rows - 1) / pad_rows * pad_rows, pre = bp[e];
    if (e % nb == b) {
      counts[e] = c;
      offsets[e] = run_u;
      pad_offsets[e] = run_p;
      const int m0 = run_p >> 7, m1 = (run_p + cp) >> 7;
      for (int m = m0; m < m1 && m < max_mtiles; ++m) mtile_expert[m] = e;
    }
    bu[e] = run_u + pre;
    bp[e] = run_p + pre;
    run_u += c;
    run_p += cp;
  }
  if (b == 0 && tid == 0) {
    offsets[E] = tot_u;
    pad_offsets[E] = tot_p;
    if ((int64_t)tot_p > rows_alloc) {
      record_status(status, MOE_DEV_CAPACITY);
      *total_mtiles = 0;
    } else {
      *total_mtiles = tot_p >> 7;
    }
  }
  // per-warp exclusive prefix of this block's counts, per expert
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int v = 0; v < kRouteWarps; ++v) {
      const int c = wh[v * E + e];
      wh[v * E + e] = run;
      run += c;
    }
  }
  __syncthreads();

  // ---- phase 3 (as route_scatter; the ids were loaded before the barrier)
  int32_t* my = wh + warp * E;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t rb = r0 + j * 32;
    if (rb >= r1) break;  // the same for the whole warp
    const int64_t r = rb + lane;
    const bool in = r < r1;
    const int id = idv[j];
    const bool act = in && id >= 0 && id < E;
    const unsigned amask = __ballot_sync(0xFFFFFFFFu, act);
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, act ? id : -1) & amask;
    int rank = 0, base = 0;
    if (act) {
      rank = __popc(peers & ((1u << lane) - 1u));
      base = my[id];
    }
    __syncwarp();
    if (act) {
      const int local = base + rank;
      const int pos = bu[id] + local;
      const int64_t ppos = (int64_t)bp[id] + local;
      perm[pos] = (int32_t)r;
      inv[r] = pos;
      inv_pad[r] = (ppos < rows_alloc) ? (int32_t)ppos : -1;
      if ((peers >> lane) == 1u) my[id] = base + __popc(peers);
    } else if (in) {
      inv[r] = -1;
      inv_pad[r] = -1;
    }
    __syncwarp();
  }
}

int route_fused_max_blocks(int E) {
  int dev = 0, coop = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
    return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  // up to 72 KB of dynamic shared memory (E = 1024)
  if (cudaFuncSetAttribute(route_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)route_fused_smem(1024)) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_fused_kernel, kFusedTokens,
                                                    route_fused_smem(E)) != cudaSuccess)
    return 0;
  return per_sm * sms;
}

cudaError_t launch_route(const Workspace& ws, const Layout& L, const int32_t* topk_idx,
                         const float* topk_w, int64_t T, bool check, cudaStream_t s,
                         cudaEvent_t const* ev, int coop_max_blocks, bool watchdog_test,
                         int64_t zero_words) {
  const int nb = (int)((T + kRouteTokens - 1) / kRouteTokens);
  const int E = L.E;
  const int max_mtiles = (int)(L.rows_alloc / 128);
  const int pad_rows = L.pad_rows > 0 ? L.pad_rows : 128;
  const int nb_fused = (int)((T + kFusedTokens - 1) / kFusedTokens);
  const bool fused = ws.grid_sync && coop_max_blocks > 0 && nb_fused <= coop_max_blocks;
  // only a one-block fused kernel clears the words itself; otherwise a memset
  if (zero_words > 0 && !(fused && nb_fused == 1) &&
      cudaMemsetAsync(ws.status, 0, (size_t)zero_words * 4, s) != cudaSuccess)
    return cudaErrorUnknown;
  if (fused) {
    if (ev) record_event(ev[0], s);
    cudaLaunchAttribute coop;
    coop.id = cudaLaunchAttributeCooperative;
    coop.val.cooperative = 1;
    const cudaError_t err = launch_k(
        route_fused_kernel, dim3(nb_fused), dim3(kFusedTokens), route_fused_smem(E), s, false, &coop,
        topk_idx, topk_w, (int)T, L.K, E, check ? 1 : 0, pad_rows, L.rows_alloc, max_mtiles,
        ws.block_counts, ws.grid_sync, ws.counts, ws.offsets, ws.pad_offsets, ws.mtile_expert,
        ws.total_mtiles, ws.perm, ws.inv, ws.inv_pad, ws.status,
        watchdog_test ? (uint64_t)20000000ull : (uint64_t)kWaitLimitNs,
        watchdog_test && nb_fused > 1 ? nb_fused - 1 : -1, ws.status,
        nb_fused == 1 ? (int)zero_words : 0);
    if (ev) {  // the scan and scatter are inside the one kernel: zero-length spans
      record_event(ev[1], s);
      record_event(ev[2], s);
    }
    return err;
  }
  if (ev) record_event(ev[0], s);
  cudaError_t err = launch_k(route_count_kernel, dim3(nb), dim3(kRouteTokens), sizeof(int32_t) * E, s,
                             false, nullptr, topk_idx, topk_w, (int)T, L.K, E, check ? 1 : 0,
                             ws.block_counts, ws.status);
  if (err != cudaSuccess) return err;
  if (ev) record_event(ev[1], s);
  err = launch_k(route_scan_kernel, dim3(1), dim3(1024), 0, s, ev == nullptr, nullptr,
                 (const int32_t*)ws.block_counts, nb, E, pad_rows, L.rows_alloc, max_mtiles, ws.counts,
                 ws.offsets, ws.pad_offsets, ws.base_u, ws.base_p, ws.mtile_expert, ws.total_mtiles,
                 ws.status);
  if (err != cudaSuccess) return err;
  if (ev) record_event(ev[2], s);
  return launch_k(route_scatter_kernel, dim3(nb), dim3(kRouteTokens), sizeof(int32_t) * 4 * E, s,
                  ev == nullptr, nullptr, topk_idx, (int)T, L.K, E, L.rows_alloc,
                  (const int32_t*)ws.base_u, (const int32_t*)ws.base_p, ws.perm, ws.inv, ws.inv_pad);
}

}  // namespace mm
