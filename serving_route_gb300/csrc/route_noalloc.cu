// route_noalloc.cu -- moe_route_noalloc: the routing step (validation,
// expert histogram, exclusive scan, stable scatter) for callers that cannot
// allocate device memory and cannot be handed a workspace.
//
// The routing kernels need scratch beyond their inputs and outputs (per-block
// histograms and bases, the padded row map, the m-tile table).  Here that
// scratch is one file-scope __device__ array of fixed size, so the call itself
// allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
// The array exists in every CUDA context that loads this library's module, for
// the life of that context.  Its device address belongs to one context: it is
// looked up on the first call made in a context (the one current on the
// calling thread, primary or not) and cached under that context's unique id.
// The kernels are the same ones moe_forward launches (route.cu); only where
// their scratch lives differs.
#include <cudaTypedefs.h>

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

// Driver entry points, through the runtime (the library does not link the
// driver library itself).
struct DriverCtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

bool driver_ctx_fns(DriverCtxFns* out) {
  static DriverCtxFns fns;
  static bool ok = false;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r1, r2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &r1) ==
            cudaSuccess &&
        r1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) ==
            cudaSuccess &&
        r2 == cudaDriverEntryPointSuccess) {
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(q);
      ok = true;
    }
  });
  *out = fns;
  return ok;
}

// Cache of the scratch address per context, keyed by the context's id (unique
// for the life of the process, so a destroyed context's entry never matches a
// later one).  Past kMaxContexts contexts the address is looked up on every
// call instead of cached.
constexpr int kMaxContexts = 64;
struct CtxScratch {
  unsigned long long ctx_id;
  int32_t* ptr;
};
CtxScratch g_ctx_scratch[kMaxContexts];
int g_ctx_count = 0;

// Device address of the scratch in the context current on this thread.
cudaError_t scratch_for_current_context(int32_t** out) {
  DriverCtxFns f;
  if (!driver_ctx_fns(&f)) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  void* p = nullptr;
  if (!ctx) {
    // No context is current on this thread yet: the runtime makes the current
    // device's primary context current when it resolves the symbol.
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    if (f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorInvalidValue;
  }
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (int i = 0; i < g_ctx_count; ++i) {
    if (g_ctx_scratch[i].ctx_id == id) {
      *out = g_ctx_scratch[i].ptr;
      return cudaSuccess;
    }
  }
  if (!p) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
  }
  if (g_ctx_count < kMaxContexts) g_ctx_scratch[g_ctx_count++] = CtxScratch{id, static_cast<int32_t*>(p)};
  *out = static_cast<int32_t*>(p);
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
  if (!d_counts || !d_offsets || !d_status) return MOE_ERR_INVALID_ARG;
  // bound num_tokens before any product is formed (no overflow below)
  if (num_tokens > kMaxRoutes) return MOE_ERR_CAPACITY;
  if (num_tokens > 0 && (!d_topk_idx || !d_topk_w || !d_perm || !d_inv)) return MOE_ERR_INVALID_ARG;
  const int64_t routes = num_tokens * top_k;
  const int64_t blocks = (num_tokens + 127) / 128;
  if (routes > kMaxRoutes || blocks * num_experts > kMaxBlockExperts) return MOE_ERR_CAPACITY;
  if (num_tokens == 0) {
    // no route: a clear status word, zero counts and offsets, nothing else
    if (cudaMemsetAsync(d_status, 0, sizeof(uint32_t), stream) != cudaSuccess ||
        cudaMemsetAsync(d_counts, 0, sizeof(int32_t) * num_experts, stream) != cudaSuccess ||
        cudaMemsetAsync(d_offsets, 0, sizeof(int32_t) * (num_experts + 1), stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }

  int32_t* scratch = nullptr;
  if (scratch_for_current_context(&scratch) != cudaSuccess) return MOE_ERR_CUDA;

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
