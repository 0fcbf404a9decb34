// route.cu -- step 1 of the layer: route validation, expert histogram,
// device-side exclusive scan and stable scatter of the routes into
// per-expert contiguous segments ("compact" in the forward diagram of
// flashinfer PR #4069; validation rules of flashinfer PR #6398 "fuse Rubin
// MegaMoE forward preparation": expert-id bounds, no duplicate routes, finite
// scores on active routes, masked slots (-1) may carry any score).
//
// Three small kernels, no host synchronisation (the second and third are
// launched as programmatic dependents, so their launch overlaps the previous
// kernel):
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
  for (int64_t rb = r0; rb < r1; rb += 32) {
    const int64_t r = rb + lane;
    const bool in = r < r1;
    const int id = in ? idx[r] : -1;
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

cudaError_t launch_route(const Workspace& ws, const Layout& L, const int32_t* topk_idx,
                         const float* topk_w, int64_t T, bool check, cudaStream_t s,
                         cudaEvent_t const* ev) {
  const int nb = (int)((T + kRouteTokens - 1) / kRouteTokens);
  const int E = L.E;
  const int max_mtiles = (int)(L.rows_alloc / 128);
  if (ev) record_event(ev[0], s);
  cudaError_t err = launch_k(route_count_kernel, dim3(nb), dim3(kRouteTokens), sizeof(int32_t) * E, s,
                             false, nullptr, topk_idx, topk_w, (int)T, L.K, E, check ? 1 : 0,
                             ws.block_counts, ws.status);
  if (err != cudaSuccess) return err;
  if (ev) record_event(ev[1], s);
  const int pad_rows = L.pad_rows > 0 ? L.pad_rows : 128;
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
