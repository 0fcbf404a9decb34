// route_noalloc.cu -- moe_route_noalloc: the routing step (validation,
// expert histogram, exclusive scan, stable scatter) for callers that cannot
// allocate device memory and cannot be handed a workspace.
//
// The routing kernels need scratch beyond their inputs and outputs (per-block
// histograms and bases, the padded row map, the m-tile table).  Here that
// scratch is one file-scope __device__ array of fixed size, so the call itself
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
// The array exists on every GPU that loads this library, for the life of the
// process.  Its device address is looked up once per device, on the first call
// made with that device current, and cached.  The kernels are the same ones
// moe_forward launches (route.cu); only where their scratch lives differs.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mm {
namespace {

// Size limits of the fixed scratch.
constexpr int64_t kMaxRoutes = 131072;        // num_tokens * top_k
constexpr int64_t kMaxBlockExperts = 32768;   // ceil(num_tokens / 128) * num_experts
constexpr int64_t kMaxExperts = 1024;
constexpr int64_t kMaxMtiles = (kMaxRoutes + 127 * kMaxExperts) / 128 + 1;

// Scratch layout in 32-bit words (each region starts on a 256-byte boundary).
constexpr int64_t kWordsAlign = 64;
constexpr int64_t up64(int64_t v) { return (v + kWordsAlign - 1) / kWordsAlign * kWordsAlign; }
constexpr int64_t kOffBlockCounts = 0;
constexpr int64_t kOffBaseU = kOffBlockCounts + up64(kMaxBlockExperts);
constexpr int64_t kOffBaseP = kOffBaseU + up64(kMaxBlockExperts);
constexpr int64_t kOffPadOffsets = kOffBaseP + up64(kMaxBlockExperts);
constexpr int64_t kOffTotalMtiles = kOffPadOffsets + up64(kMaxExperts + 1);
constexpr int64_t kOffMtileExpert = kOffTotalMtiles + kWordsAlign;
constexpr int64_t kOffInvPad = kOffMtileExpert + up64(kMaxMtiles);
constexpr int64_t kScratchWords = kOffInvPad + up64(kMaxRoutes);

// The scratch itself: about 0.9 MiB of device memory per GPU.
static __device__ __align__(256) int32_t g_route_scratch[kScratchWords];

std::mutex g_scratch_mu;
constexpr int kMaxDevices = 64;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch for the current device (looked up once).
cudaError_t scratch_for_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mm

using namespace mm;

extern "C" moe_status moe_route_noalloc(const int32_t* d_topk_idx, const float* d_topk_w,
                                        int64_t num_tokens, int32_t top_k, int32_t num_experts,
                                        int32_t check_routes, int32_t* d_counts,
                                        int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv,
                                        uint32_t* d_status, struct CUstream_st* stream) {
  const bool k_ok = top_k == 1 || top_k == 2 || top_k == 4 || top_k == 6 || top_k == 8;
  if (!k_ok || num_experts < 1 || num_experts > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (num_tokens < 0) return MOE_ERR_INVALID_ARG;
  if (num_tokens == 0) return MOE_OK;
  if (!d_topk_idx || !d_topk_w || !d_counts || !d_offsets || !d_perm || !d_inv || !d_status)
    return MOE_ERR_INVALID_ARG;
  const int64_t routes = num_tokens * top_k;
  const int64_t blocks = (num_tokens + 127) / 128;
  if (routes > kMaxRoutes || blocks * num_experts > kMaxBlockExperts) return MOE_ERR_CAPACITY;

  int32_t* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;

  Layout L;
  memset(&L, 0, sizeof(L));
  L.E = num_experts;
  L.K = top_k;
  L.max_rows = num_tokens;
  const int64_t padded = routes + 127 * (routes < num_experts ? routes : (int64_t)num_experts);
  L.rows_alloc = (padded + 127) / 128 * 128;

  Workspace ws;
  memset(&ws, 0, sizeof(ws));
  ws.status = d_status;
  ws.counts = d_counts;
  ws.offsets = d_offsets;
  ws.perm = d_perm;
  ws.inv = d_inv;
  ws.block_counts = scratch + kOffBlockCounts;
  ws.base_u = scratch + kOffBaseU;
  ws.base_p = scratch + kOffBaseP;
  ws.pad_offsets = scratch + kOffPadOffsets;
  ws.total_mtiles = scratch + kOffTotalMtiles;
  ws.mtile_expert = scratch + kOffMtileExpert;
  ws.inv_pad = scratch + kOffInvPad;

  // Nothing in the scratch needs clearing: every entry a call reads was
  // written earlier in the same call.  The caller's status word is cleared
  // here because the kernels OR error bits into it.
  if (cudaMemsetAsync(d_status, 0, sizeof(uint32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
  // the three-kernel routing: the cooperative one-kernel form would need a
  // zeroed arrival counter in the scratch
  if (launch_route(ws, L, d_topk_idx, d_topk_w, num_tokens, check_routes != 0, stream, nullptr,
                   0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
