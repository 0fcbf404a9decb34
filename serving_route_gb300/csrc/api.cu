// api.cu -- the C ABI (include/megamoe.h): argument checks, workspace and
// weight-store layout, TMA tensor-map encoding, and the stream-ordered launch
// sequence of one forward.  The calls follow the problem statement of
// flashinfer PR #4069 ("Contracts introduced by this PR": capacity-bounded
// workspace query with expected_m / max_rows, construction binding
// transformed static weights, stage_inputs pre-binding the output) and the
// tail-masking convention of flashinfer PR #6398.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "common.cuh"
#include "internal.h"

using namespace mm;

struct moe_handle {
  moe_dims dims;
  Layout L;
  int64_t expected_m;
  Workspace ws;
  WeightStore wst;
  CUtensorMap tm_a, tm_hq;                  // blocked activations: one 128x128 box per load
  CUtensorMap tm_a_sw[3], tm_hq_sw[3];      // the same with 16 / 32 / 64-row boxes (token-as-N GEMMs)
  CUtensorMap tm_w1, tm_w2;                 // blocked weights: one 128x128 box per load
  CUtensorMap tm_asf, tm_hsf;               // scale atoms as 2-D uint32 tensors (CTA pairs)
  CUtensorMap tm_w1sf, tm_w2sf;             // weight scale atoms, same form (CTA pairs)
  CUtensorMap tm_y;                         // FC2 output, 32x32 BF16 boxes (TMA stores)
  int pair_ctas;                            // grid of the CTA-pair GEMMs
  int sm_budget;                            // moe_set_sm_budget (0: every SM)
  int route_coop_blocks;                    // co-resident grid limit of the one-kernel routing
  int quant_resident[2];                    // resident blocks of quant_dispatch, 2 / 4 units per pass
  bool bound;
  bool pt_scales;                           // per-tensor: activation scales given
  float pt_x_scale, pt_h_scale;
  uint16_t* out;
  int num_sms;
  int device;
  cudaEvent_t ev[10];
  int n_ev;
};

namespace {

constexpr size_t kAlign = 1024;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool valid_dims(const moe_dims* d) {
  if (!d) return false;
  const bool hk = d->hidden >= 128 && d->hidden <= 16384 && d->hidden % 128 == 0;
  const bool ik = d->inter >= 128 && d->inter <= 16384 && d->inter % 128 == 0;
  const bool ek = d->num_experts >= 1 && d->num_experts <= 1024;
  const bool kk = d->top_k == 1 || d->top_k == 2 || d->top_k == 4 || d->top_k == 6 || d->top_k == 8;
  return hk && ik && ek && kk;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// BF16 matrix [rows, cols] for TMA stores of 32-row x 32-column boxes,
// 64-byte swizzle.
bool encode_bf16_store_map(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Blocked weight store [row blocks][kblocks][128 rows][128 B] as a 3-D byte
// tensor {128, kblocks * 128, row blocks}; box {128, 128, 1} = one contiguous
// 16 KB block, 128-byte swizzle.
// box_rows < 128: the first box_rows rows of a block (the token tiles of the
// token-as-N GEMMs).
bool encode_blocked_map(CUtensorMap* m, const void* base, uint64_t kblocks, uint64_t row_blocks,
                        uint32_t box_rows = 128,
                        CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, kblocks * 128, row_blocks};
  cuuint64_t strides[2] = {128, kblocks * 128 * 128};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale atoms [n_atoms][512 B] as a 2-D uint32 tensor [n_atoms, 128]; one
// atom per box, no swizzle.
bool encode_atom_map(CUtensorMap* m, const void* base, uint64_t n_atoms) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, n_atoms};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// SMs a forward may occupy, and the GEMM grid that follows from it.
int budget_sms(const moe_handle* h) {
  return (h->sm_budget > 0 && h->sm_budget < h->num_sms) ? h->sm_budget : h->num_sms;
}

// Tile rounds of a forward of T tokens, estimated on the host (the real
// counts stay on the device): routed rows per touched expert, padded to the
// tactic's segment, in 128-row m-tiles, times the FC1 + FC2 n-tiles, over the
// GEMM grid (in pairs for CTA pairs).
double gemm_rounds_estimate(const moe_handle* h, int grid, int64_t T) {
  const Layout& L = h->L;
  const double routes = (double)T * L.K;
  const double touched = routes < L.E ? routes : (double)L.E;
  const double per = routes / touched;
  const double seg = std::ceil(per / L.pad_rows) * L.pad_rows;
  const double mtiles = touched * seg / 128.0;
  const double units = (L.pair ? mtiles / 2 : mtiles) * (L.I / 128 + (L.H + 255) / 256);
  const double slots = L.pair ? grid / 2 : grid;
  return units / (slots > 0 ? slots : 1);
}

int gemm_grid(const moe_handle* h) {
  const int sms = budget_sms(h);
  if (!h->L.pair) return sms;
  const int c = sms & ~1;
  return c < h->pair_ctas ? c : h->pair_ctas;
}

// What a forward of T tokens launches (without profiling events): one
// cooperative routing kernel when its blocks can all be resident and no SM
// budget is set; FC1 -> FC2 as one launch when the fused epilogue is on and
// the forward is short (or forced).
// Token tile of the token-as-N GEMMs for a forward of T tokens (0: the
// M128 x N256 kernel): single-CTA tactic, not switched off, and T <= 64, so
// that no expert has more routed rows than the tile.
int swap_tokens(const moe_handle* h, int64_t T) {
  if (h->L.pair || (h->dims.flags & MOE_FLAG_NO_SWAP_AB) || T <= 0) return 0;
  return T <= 16 ? 16 : (T <= 32 ? 32 : (T <= 64 ? 64 : 0));
}

moe_plan forward_plan(const moe_handle* h, int64_t T) {
  moe_plan p = {0, 0, 0, 0, 0, 0};
  if (T <= 0) return p;
  const uint32_t f = h->dims.flags;
  const bool fused = (f & MOE_FLAG_FUSE_FC1_EPILOGUE) != 0;
  const int64_t fused_blocks = (T + 511) / 512;
  const int coop = h->sm_budget > 0 ? 0 : h->route_coop_blocks;
  p.route_kernels = (coop > 0 && fused_blocks <= coop) ? 1 : 3;
  const bool one = fused && !(f & MOE_FLAG_SPLIT_GEMMS) &&
                   ((f & MOE_FLAG_GEMMS_ONE_LAUNCH) || gemm_rounds_estimate(h, gemm_grid(h), T) <= 48.0);
  p.gemm_launches = one ? 1 : 2;
  p.swiglu_kernels = fused ? 0 : 1;
  p.swap_ab_tokens = swap_tokens(h, T);
  // single-CTA FC2 launches (token-as-N or M128 x N256) fold the combine in
  // when asked to; CTA pairs keep the combine kernel
  p.combine_in_fc2 = (!h->L.pair && (f & MOE_FLAG_COMBINE_IN_FC2)) ? 1 : 0;
  p.kernels = p.route_kernels + 1 + p.gemm_launches + p.swiglu_kernels + (p.combine_in_fc2 ? 0 : 1);
  return p;
}

}  // namespace

namespace mm {

moe_status compute_layout(const moe_dims* d, int64_t expected_m, int64_t max_rows, float cf,
                          Layout* L) {
  if (!valid_dims(d)) return MOE_ERR_UNSUPPORTED;
  if ((d->flags & MOE_FLAG_SPLIT_GEMMS) && (d->flags & MOE_FLAG_GEMMS_ONE_LAUNCH))
    return MOE_ERR_INVALID_ARG;
  if ((d->flags & MOE_FLAG_GEMM_SINGLE_CTA) && (d->flags & MOE_FLAG_GEMM_CTA_PAIR))
    return MOE_ERR_INVALID_ARG;
  if (max_rows < 1 || max_rows > (int64_t)1 << 24) return MOE_ERR_INVALID_ARG;
  if (!(cf > 0.f) || !(cf <= 64.f)) return MOE_ERR_INVALID_ARG;
  memset(L, 0, sizeof(*L));
  L->H = d->hidden;
  L->I = d->inter;
  L->E = d->num_experts;
  L->K = d->top_k;
  L->max_rows = max_rows;
  // tactic (flashinfer PR #4069, Contracts: expected_m selects the tactic and
  // max_rows / capacity_factor the memory bound, independently).
  // A CTA pair (M = 256 over two SMs) stages 32 KB per K block and SM instead
  // of 48 KB, so on GB300 it keeps the tensor cores fed ~13% better per
  // GEMM row; but it pads every expert segment to 256 rows instead of 128.
  // Automatic choice: with m = expected_m * K / E routed rows per expert,
  // pairs when their padded rows cost less than 1.13x the single-CTA rows.
  const bool force_single = (d->flags & MOE_FLAG_GEMM_SINGLE_CTA) != 0;
  const bool force_pair = (d->flags & MOE_FLAG_GEMM_CTA_PAIR) != 0;
  bool pair = force_pair;
  if (!force_single && !force_pair) {
    const double m = (double)expected_m * d->top_k / d->num_experts;
    const double single_rows = std::ceil(m / 128.0) * 128.0, pair_rows = std::ceil(m / 256.0) * 256.0;
    pair = pair_rows < 1.13 * single_rows;
  }
  L->pair = pair;
  L->pad_rows = pair ? 256 : 128;
  // buffers are sized for the padding of any tactic the flags allow, so the
  // sizes never depend on expected_m
  const int64_t size_pad = force_single ? 128 : 256;
  const int64_t rk = max_rows * L->K;
  int64_t cap = (int64_t)std::ceil((double)cf * (double)rk);
  if (cap > rk) cap = rk;
  if (cap < 1) cap = 1;
  L->cap_rows = cap;
  // capacity: routed rows plus at most pad_rows - 1 padding rows per non-empty
  // expert (buffer sizes depend on max_rows, capacity_factor and the flags,
  // never on expected_m)
  const int64_t pad = cap + (size_pad - 1) * (cap < L->E ? cap : (int64_t)L->E);
  L->rows_alloc = (int64_t)align_up((size_t)(pad < size_pad ? size_pad : pad), (size_t)size_pad);
  if (L->rows_alloc > ((int64_t)1 << 31) - 256) return MOE_ERR_INVALID_ARG;
  L->nb_max = (max_rows + 127) / 128;
  L->keep_gu = !(d->flags & MOE_FLAG_FUSE_FC1_EPILOGUE) || (d->flags & MOE_FLAG_EMIT_FC1);
  L->mx = (d->flags & MOE_FLAG_MXFP8) != 0;
  L->pt = (d->flags & MOE_FLAG_PER_TENSOR) != 0;
  if (L->mx && L->pt) return MOE_ERR_INVALID_ARG;
  const size_t H = L->H, I = L->I, E = L->E, R = L->rows_alloc, MB = R / 128;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, kAlign);
    return at;
  };
  // status word at +0, total_mtiles at +4, routing arrival counter at +8;
  // the megakernel's per-m-tile counters follow at +1024, so one memset
  // clears both
  // the folded combine's counters ([max_rows tokens][ceil(H/256)]) follow
  // the per-m-tile counters, under the same memset
  const size_t cmb_bytes = 4 * (size_t)max_rows * ((H + 255) / 256);
  L->o_status = take(1024 + 4 * MB + cmb_bytes);
  L->o_fc1_done = L->o_status + 1024;
  L->o_cmb = L->o_fc1_done + 4 * MB;
  L->o_counts = take(4 * E);
  L->o_offsets = take(4 * (E + 1));
  L->o_pad_offsets = take(4 * (E + 1));
  L->o_mtile_expert = take(4 * MB);
  L->o_block_counts = take(4 * (size_t)L->nb_max * E);
  L->o_base_u = take(4 * (size_t)L->nb_max * E);
  L->o_base_p = take(4 * (size_t)L->nb_max * E);
  L->o_perm = take(4 * (size_t)rk);
  L->o_inv = take(4 * (size_t)rk);
  L->o_inv_pad = take(4 * (size_t)rk);
  L->o_a = take(R * H);
  L->o_a_sf = take(MB * atoms_along_k(H / 128, L->mx) * kSfAtomBytes);
  L->o_gu = L->keep_gu ? take(R * 2 * I * 2) : 0;
  L->o_hq = take(R * I);
  L->o_h_sf = take(MB * atoms_along_k(I / 128, L->mx) * kSfAtomBytes);
  L->o_y = take(R * H * 2);
  L->ws_bytes = o + kAlign;  // slack to align the caller's base
  o = 0;
  L->o_w1 = take(E * 2 * I * H);
  L->o_w2 = take(E * H * I);
  L->o_w1_sf = take(E * (2 * I / 128) * (H / 128));
  L->o_w2_sf = take(E * (H / 128) * (I / 128));
  L->o_w1_sfatoms = take(E * (2 * I / 128) * atoms_along_k(H / 128, L->mx) * kSfAtomBytes);
  L->o_w2_sfatoms = take(E * (H / 128) * atoms_along_k(I / 128, L->mx) * kSfAtomBytes);
  L->o_pt = L->pt ? take(4 * (4 * E + 2)) : 0;
  L->w_bytes = o + kAlign;
  return MOE_OK;
}

}  // namespace mm

extern "C" {

moe_status moe_workspace_query(const moe_dims* dims, int64_t expected_m, int64_t max_rows,
                               float capacity_factor, size_t* workspace_bytes,
                               size_t* weight_bytes) {
  if (!dims || !workspace_bytes || !weight_bytes) return MOE_ERR_INVALID_ARG;
  if (expected_m < 1) return MOE_ERR_INVALID_ARG;
  Layout L;
  const moe_status st = compute_layout(dims, expected_m, max_rows, capacity_factor, &L);
  if (st != MOE_OK) return st;
  *workspace_bytes = L.ws_bytes;
  *weight_bytes = L.w_bytes;
  return MOE_OK;
}

moe_status moe_create(const moe_dims* dims, int64_t expected_m, int64_t max_rows,
                      float capacity_factor, void* d_workspace, size_t workspace_bytes,
                      void* d_weight_store, size_t weight_bytes, moe_handle** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!dims || !d_workspace || !d_weight_store || expected_m < 1) return MOE_ERR_INVALID_ARG;
  Layout L;
  moe_status st = compute_layout(dims, expected_m, max_rows, capacity_factor, &L);
  if (st != MOE_OK) return st;
  if (workspace_bytes < L.ws_bytes || weight_bytes < L.w_bytes) return MOE_ERR_WORKSPACE;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  if (gemm_set_attributes() != cudaSuccess || gemm_swap_set_attributes() != cudaSuccess)
    return MOE_ERR_CUDA;
  moe_handle* h = new (std::nothrow) moe_handle;
  if (!h) return MOE_ERR_INVALID_ARG;
  memset(h, 0, sizeof(*h));
  h->dims = *dims;
  h->L = L;
  h->expected_m = expected_m;
  h->num_sms = sms;
  h->route_coop_blocks = route_fused_max_blocks(L.E);
  const int fmt = L.pt ? 2 : (L.mx ? 1 : 0);
  h->quant_resident[0] = quant_dispatch_resident(fmt, 2);
  h->quant_resident[1] = quant_dispatch_resident(fmt, 4);
  h->device = dev;
  uint8_t* b = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(d_workspace), kAlign));
  Workspace& w = h->ws;
  w.status = reinterpret_cast<uint32_t*>(b + L.o_status);
  w.total_mtiles = reinterpret_cast<int32_t*>(b + L.o_status + 4);
  w.grid_sync = reinterpret_cast<uint32_t*>(b + L.o_status + 8);
  w.gemm_sched = reinterpret_cast<int32_t*>(b + L.o_status + 12);
  w.fc1_done = reinterpret_cast<int32_t*>(b + L.o_fc1_done);
  w.cmb_cnt = reinterpret_cast<int32_t*>(b + L.o_cmb);
  w.counts = reinterpret_cast<int32_t*>(b + L.o_counts);
  w.offsets = reinterpret_cast<int32_t*>(b + L.o_offsets);
  w.pad_offsets = reinterpret_cast<int32_t*>(b + L.o_pad_offsets);
  w.mtile_expert = reinterpret_cast<int32_t*>(b + L.o_mtile_expert);
  w.block_counts = reinterpret_cast<int32_t*>(b + L.o_block_counts);
  w.base_u = reinterpret_cast<int32_t*>(b + L.o_base_u);
  w.base_p = reinterpret_cast<int32_t*>(b + L.o_base_p);
  w.perm = reinterpret_cast<int32_t*>(b + L.o_perm);
  w.inv = reinterpret_cast<int32_t*>(b + L.o_inv);
  w.inv_pad = reinterpret_cast<int32_t*>(b + L.o_inv_pad);
  w.a = b + L.o_a;
  w.a_sf = b + L.o_a_sf;
  w.gu = L.keep_gu ? reinterpret_cast<uint16_t*>(b + L.o_gu) : nullptr;
  w.hq = b + L.o_hq;
  w.h_sf = b + L.o_h_sf;
  w.y = reinterpret_cast<uint16_t*>(b + L.o_y);
  uint8_t* wb =
      reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(d_weight_store), kAlign));
  h->wst.w1 = wb + L.o_w1;
  h->wst.w2 = wb + L.o_w2;
  h->wst.w1_sf = wb + L.o_w1_sf;
  h->wst.w2_sf = wb + L.o_w2_sf;
  h->wst.w1_sfatoms = wb + L.o_w1_sfatoms;
  h->wst.w2_sfatoms = wb + L.o_w2_sfatoms;
  h->wst.pt = L.pt ? reinterpret_cast<float*>(wb + L.o_pt) : nullptr;
  if (!encode_blocked_map(&h->tm_a, w.a, L.H / 128, (uint64_t)(L.rows_alloc / 128)) ||
      !encode_blocked_map(&h->tm_hq, w.hq, L.I / 128, (uint64_t)(L.rows_alloc / 128)) ||
      !encode_atom_map(&h->tm_asf, w.a_sf, (uint64_t)(L.rows_alloc / 128) * atoms_along_k(L.H / 128, L.mx)) ||
      !encode_atom_map(&h->tm_hsf, w.h_sf, (uint64_t)(L.rows_alloc / 128) * atoms_along_k(L.I / 128, L.mx)) ||
      !encode_atom_map(&h->tm_w1sf, h->wst.w1_sfatoms,
                       (uint64_t)L.E * (2 * L.I / 128) * atoms_along_k(L.H / 128, L.mx)) ||
      !encode_atom_map(&h->tm_w2sf, h->wst.w2_sfatoms,
                       (uint64_t)L.E * (L.H / 128) * atoms_along_k(L.I / 128, L.mx)) ||
      !encode_bf16_store_map(&h->tm_y, w.y, L.H, L.rows_alloc) ||
      !encode_blocked_map(&h->tm_a_sw[0], w.a, L.H / 128, (uint64_t)(L.rows_alloc / 128), 16) ||
      !encode_blocked_map(&h->tm_a_sw[1], w.a, L.H / 128, (uint64_t)(L.rows_alloc / 128), 32) ||
      !encode_blocked_map(&h->tm_a_sw[2], w.a, L.H / 128, (uint64_t)(L.rows_alloc / 128), 64) ||
      !encode_blocked_map(&h->tm_hq_sw[0], w.hq, L.I / 128, (uint64_t)(L.rows_alloc / 128), 16) ||
      !encode_blocked_map(&h->tm_hq_sw[1], w.hq, L.I / 128, (uint64_t)(L.rows_alloc / 128), 32) ||
      !encode_blocked_map(&h->tm_hq_sw[2], w.hq, L.I / 128, (uint64_t)(L.rows_alloc / 128), 64)) {
    delete h;
    return MOE_ERR_CUDA;
  }
  if (h->L.pair) {
    const int pairs = gemm_max_pairs();
    if (pairs <= 0)
      h->L.pair = false;  // no co-resident CTA pairs: single-CTA kernel on the same layout
    else
      h->pair_ctas = 2 * pairs;
  }
  *out = h;
  return MOE_OK;
}

moe_status moe_quantize_weights(const float* d_w, int64_t num_mats, int32_t rows, int32_t cols,
                                uint8_t* d_q, float* d_scale, struct CUstream_st* stream) {
  if (!d_w || !d_q || !d_scale || num_mats < 0 || rows <= 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (rows % 128 || cols % 128) return MOE_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(d_w) % 16 || reinterpret_cast<uintptr_t>(d_q) % 16)
    return MOE_ERR_INVALID_ARG;
  if (launch_quantize_weights(d_w, num_mats, rows, cols, d_q, d_scale, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_requantize_weights_nvfp4(const uint8_t* d_codes, const uint8_t* d_block_scales,
                                        const float* d_global_scales, int64_t num_mats, int32_t rows,
                                        int32_t cols, uint8_t* d_q, float* d_scale,
                                        struct CUstream_st* stream) {
  if (!d_codes || !d_block_scales || !d_global_scales || !d_q || !d_scale || num_mats < 0 ||
      rows <= 0 || cols <= 0)
    return MOE_ERR_INVALID_ARG;
  if (rows % 128 || cols % 128) return MOE_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(d_codes) % 16 || reinterpret_cast<uintptr_t>(d_block_scales) % 4 ||
      reinterpret_cast<uintptr_t>(d_q) % 16)
    return MOE_ERR_INVALID_ARG;
  if (launch_requant_nvfp4(d_codes, d_block_scales, d_global_scales, num_mats, rows, cols, d_q,
                           d_scale, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_quantize_weights_mx(const float* d_w, int64_t num_mats, int32_t rows, int32_t cols,
                                   uint8_t* d_q, float* d_scale, struct CUstream_st* stream) {
  if (!d_w || !d_q || !d_scale || num_mats < 0 || rows <= 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (rows % 128 || cols % 128) return MOE_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(d_w) % 16 || reinterpret_cast<uintptr_t>(d_q) % 16)
    return MOE_ERR_INVALID_ARG;
  if (launch_quantize_weights_mx(d_w, num_mats, rows, cols, d_q, d_scale, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_quantize_weights_pt(const float* d_w, int64_t num_mats, int32_t rows, int32_t cols,
                                   uint8_t* d_q, float* d_scale, struct CUstream_st* stream) {
  if (!d_w || !d_q || !d_scale || num_mats < 0 || rows <= 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (rows % 128 || cols % 128) return MOE_ERR_UNSUPPORTED;
  if (num_mats > 65535) return MOE_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(d_w) % 16 || reinterpret_cast<uintptr_t>(d_q) % 16 ||
      reinterpret_cast<uintptr_t>(d_scale) % 4)
    return MOE_ERR_INVALID_ARG;
  if (launch_quantize_weights_pt(d_w, num_mats, rows, cols, d_q, d_scale, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_set_activation_scales(moe_handle* h, float x_scale, float h_scale,
                                     struct CUstream_st* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (!h->L.pt) return MOE_ERR_UNSUPPORTED;
  if (!(x_scale > 0.f) || !std::isfinite(x_scale) || !(h_scale > 0.f) || !std::isfinite(h_scale))
    return MOE_ERR_INVALID_ARG;
  h->pt_x_scale = x_scale;
  h->pt_h_scale = h_scale;
  h->pt_scales = true;
  // the epilogue factors need the bound weight scales; before the bind they
  // are computed there
  if (h->bound && launch_pt_set_scales(h->wst, h->L, x_scale, h_scale, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_bind_weights(moe_handle* h, const uint8_t* d_w1, const float* d_w1_scale,
                            const uint8_t* d_w2, const float* d_w2_scale,
                            struct CUstream_st* stream) {
  if (!h || !d_w1 || !d_w1_scale || !d_w2 || !d_w2_scale) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_w1) % 16) return MOE_ERR_INVALID_ARG;
  h->bound = false;
  const Layout& L = h->L;
  if (cudaMemsetAsync(h->ws.status, 0, 4, stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_bind_transform(h->wst, L, d_w1, d_w1_scale, d_w2, d_w2_scale, h->ws.status, stream) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (L.pt && h->pt_scales &&
      launch_pt_set_scales(h->wst, L, h->pt_x_scale, h->pt_h_scale, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  uint32_t st = 0;
  if (cudaMemcpyAsync(&st, h->ws.status, 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (st & MOE_DEV_BAD_SCALE) return MOE_ERR_BAD_SCALE;
  // weight boxes are contiguous 16 KB runs read once per tile: no L2
  // promotion (decode T = 256: 1.6563 -> 1.6544 ms against 256-byte promotion)
  if (!encode_blocked_map(&h->tm_w1, h->wst.w1, L.H / 128, (uint64_t)L.E * (2 * L.I / 128), 128,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
      !encode_blocked_map(&h->tm_w2, h->wst.w2, L.I / 128, (uint64_t)L.E * (L.H / 128), 128,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return MOE_ERR_CUDA;
  h->bound = true;
  return MOE_OK;
}

moe_status moe_stage_inputs(moe_handle* h, uint16_t* d_out) {
  if (!h || !d_out) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_out) % 16) return MOE_ERR_INVALID_ARG;
  h->out = d_out;
  return MOE_OK;
}

moe_status moe_forward(moe_handle* h, const uint16_t* d_x, const int32_t* d_topk_idx,
                       const float* d_topk_w, int64_t num_tokens, struct CUstream_st* stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (!h->bound || !h->out || (h->L.pt && !h->pt_scales)) return MOE_ERR_NOT_BOUND;
  if (num_tokens < 0) return MOE_ERR_INVALID_ARG;
  if (num_tokens > h->L.max_rows) return MOE_ERR_CAPACITY;
  if (num_tokens == 0) return MOE_OK;
  if (!d_x || !d_topk_idx || !d_topk_w) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_x) % 16) return MOE_ERR_INVALID_ARG;
  const Layout& L = h->L;
  const Workspace& ws = h->ws;
  cudaStream_t s = stream;
  const cudaEvent_t* ev = h->n_ev ? h->ev : nullptr;
  const bool fused = (h->dims.flags & MOE_FLAG_FUSE_FC1_EPILOGUE) != 0;
  const bool emit = (h->dims.flags & MOE_FLAG_EMIT_FC1) != 0;
  const bool check = (h->dims.flags & MOE_FLAG_CHECK_ROUTES) != 0;

  if (ev) record_event(ev[0], s);
  // Both GEMMs in one launch unless asked otherwise or profiled per kernel
  // (events between kernels need two launches to time FC1 and FC2).
  const moe_plan plan = forward_plan(h, num_tokens);
  const bool mega = ev == nullptr && plan.gemm_launches == 1;
  // status word, total_mtiles, the routing kernel's arrival counter, the
  // GEMM launches' unit counters and (for the megakernel) the per-m-tile FC1
  // counters
  // (and, with the combine folded into FC2, the counters of this forward's tokens)
  const bool fold = plan.combine_in_fc2 != 0;
  const size_t reset = fold ? L.o_cmb - L.o_status + 4 * (size_t)num_tokens * ((L.H + 255) / 256)
                            : (mega ? 1024 + 4 * (size_t)(L.rows_alloc / 128) : 20);
  // A one-block routing kernel (the one-kernel form, at most 512 tokens)
  // clears them itself, which saves the forward a memset node.
  const bool route_clears = plan.route_kernels == 1 && num_tokens <= 512;
  if (!route_clears && cudaMemsetAsync(ws.status, 0, reset, s) != cudaSuccess) return MOE_ERR_CUDA;
  // Under an SM budget the routing keeps to its three small kernels: a
  // cooperative grid would have to be resident beside the side-stream work.
  const int coop = plan.route_kernels == 1 ? h->route_coop_blocks : 0;
  if (launch_route(ws, L, d_topk_idx, d_topk_w, num_tokens, check, s, ev ? ev + 1 : nullptr,
                   coop, (h->dims.flags & MOE_FLAG_WATCHDOG_ROUTE_TEST) != 0,
                   route_clears ? (int64_t)(reset / 4) : 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ev) record_event(ev[4], s);
  // Kernels after the first are programmatic dependents of their predecessor
  // unless profiling events sit between them.
  const bool pdl = ev == nullptr;
  // streaming kernels: up to 16 CTAs per SM, or one per SM of the budget
  // Streaming kernels keep their full grids under an SM budget: their CTAs
  // cannot be confined to a subset of SMs, and one CTA per budgeted SM
  // starves them of memory parallelism.  The budget caps the persistent GEMM.
  const int stream_ctas = 16 * h->num_sms;
  // per-tensor: the reciprocals and per-expert factors in the weight store
  const float* pt_rx = L.pt ? h->wst.pt + 4 * L.E : nullptr;
  const float* pt_rh = L.pt ? h->wst.pt + 4 * L.E + 1 : nullptr;
  if (launch_quant_dispatch(ws, L, d_x, num_tokens, s, pdl, stream_ctas, h->quant_resident[0],
                            h->quant_resident[1], pt_rx) != cudaSuccess)
    return MOE_ERR_CUDA;

  GemmArgs g1;
  memset(&g1, 0, sizeof(g1));
  g1.sfa = ws.a_sf;
  g1.sfb = h->wst.w1_sfatoms;
  g1.mtile_expert = ws.mtile_expert;
  g1.total_mtiles = ws.total_mtiles;
  g1.counts = ws.counts;
  g1.pad_offsets = ws.pad_offsets;
  g1.KB = L.H / 128;
  g1.KQ = (int)atoms_along_k(g1.KB, L.mx);
  g1.mx = L.mx ? 1 : 0;
  g1.NT = L.I / 128;  // 256-wide tiles over 2I
  g1.N = 2 * L.I;
  g1.NB = 2 * L.I / 128;
  g1.max_mtiles = (int)(L.rows_alloc / 128);
  g1.out = ws.gu;
  g1.ld_out = 2 * (int64_t)L.I;
  g1.inter = L.I;
  g1.hq = ws.hq;
  g1.h_sf = ws.h_sf;
  g1.IB = L.I / 128;
  g1.status = ws.status;
  const bool wd_test = (h->dims.flags & MOE_FLAG_WATCHDOG_TEST) != 0;
  g1.wait_limit_ns = wd_test ? 20000000ull : 1000000000ull;
  g1.watchdog_test = wd_test ? 1 : 0;
  // Single CTAs take units from a counter when the forward routes fewer rows
  // than one full 128-row m-tile per expert: its tiles then mostly stream
  // weights and their durations vary with memory contention (and FC1 units
  // cost several FC2 units), which the counter evens out (decode T = 8:
  // 0.3745 -> 0.3634 ms).  With full m-tiles the tiles are compute-shaped and
  // of equal cost, the static round robin is already balanced and the
  // counter only adds jitter (dsv2lite: 0.2591 -> 0.2650 ms).  CTA pairs
  // keep the static order.
  const bool dyn_sched = !L.pair && num_tokens * L.K < 128 * (int64_t)L.E;
  g1.sched = dyn_sched ? ws.gemm_sched : nullptr;
  g1.pt_scale = L.pt ? h->wst.pt + 2 * L.E : nullptr;
  g1.pt_rh = pt_rh;
  const GemmMode m1 = fused ? (emit ? kModeFusedGU : kModeFused) : kModeGU;
  if (ev) record_event(ev[5], s);
  const bool pair = L.pair;
  const int ctas = gemm_grid(h);
  // token-as-N GEMMs for small forwards: the maps whose box is the token tile
  const int swap = plan.swap_ab_tokens;
  const int si = swap == 16 ? 0 : (swap == 32 ? 1 : 2);
  if (!mega && swap &&
      launch_gemm_swap(m1, swap, &h->tm_a_sw[si], &h->tm_w1, &h->tm_a_sw[si], &h->tm_w1, g1, g1, ctas,
                       s, pdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!mega && !swap &&
      launch_gemm(m1, pair, &h->tm_a, &h->tm_w1, &h->tm_asf, &h->tm_w1sf, &h->tm_y, g1, ctas, s,
                  pdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ev) record_event(ev[6], s);
  if (!fused && launch_swiglu_quant(ws, L, stream_ctas, s, pdl, pt_rh) != cudaSuccess)
    return MOE_ERR_CUDA;

  GemmArgs g2;
  memset(&g2, 0, sizeof(g2));
  g2.sfa = ws.h_sf;
  g2.sfb = h->wst.w2_sfatoms;
  g2.mtile_expert = ws.mtile_expert;
  g2.total_mtiles = ws.total_mtiles;
  g2.counts = ws.counts;
  g2.pad_offsets = ws.pad_offsets;
  g2.KB = L.I / 128;
  g2.KQ = (int)atoms_along_k(g2.KB, L.mx);
  g2.mx = L.mx ? 1 : 0;
  g2.NT = (L.H + 255) / 256;
  g2.N = L.H;
  g2.NB = L.H / 128;
  g2.max_mtiles = (int)(L.rows_alloc / 128);
  g2.out = ws.y;
  g2.ld_out = L.H;
  g2.status = ws.status;
  g2.wait_limit_ns = g1.wait_limit_ns;
  g2.sched = dyn_sched ? ws.gemm_sched + 1 : nullptr;
  g2.pt_scale = L.pt ? h->wst.pt + 3 * L.E : nullptr;
  if (fold) {
    g2.cmb_cnt = ws.cmb_cnt;
    g2.cmb_out = h->out;
    g2.cmb_w = d_topk_w;
    g2.cmb_inv = ws.inv_pad;
    g2.cmb_perm = ws.perm;
    g2.cmb_offsets = ws.offsets;
    g2.cmb_T = (int)num_tokens;
    g2.cmb_K = L.K;
  }
  if (ev) record_event(ev[7], s);
  if (mega) {
    // the FC1 epilogue publishes, per m-tile, how many of its NT tiles are stored
    g2.fc1_done = ws.fc1_done;
    g2.fc1_ntiles = g1.NT;
    g1.fc1_done = ws.fc1_done;
    g1.fc1_ntiles = g1.NT;
    const cudaError_t e =
        swap ? launch_gemm_swap(kModeMega, swap, &h->tm_a_sw[si], &h->tm_w1, &h->tm_hq_sw[si],
                                &h->tm_w2, g1, g2, ctas, s, pdl)
             : launch_gemm_mega(pair, &h->tm_a, &h->tm_w1, &h->tm_asf, &h->tm_w1sf, &h->tm_hq,
                                &h->tm_w2, &h->tm_hsf, &h->tm_w2sf, &h->tm_y, g1, g2, ctas, s, pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    const cudaError_t e =
        swap ? launch_gemm_swap(kModeY, swap, &h->tm_hq_sw[si], &h->tm_w2, &h->tm_hq_sw[si],
                                &h->tm_w2, g2, g2, ctas, s, pdl)
             : launch_gemm(kModeY, pair, &h->tm_hq, &h->tm_w2, &h->tm_hsf, &h->tm_w2sf, &h->tm_y, g2,
                           ctas, s, pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (ev) record_event(ev[8], s);
  if (!fold && launch_combine(ws, L, d_topk_w, h->out, num_tokens, s, pdl, stream_ctas) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ev) record_event(ev[9], s);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_read_status(moe_handle* h, uint32_t* h_status, struct CUstream_st* stream) {
  if (!h || !h_status) return MOE_ERR_INVALID_ARG;
  uint32_t st = 0;
  if (cudaMemcpyAsync(&st, h->ws.status, 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  *h_status = st;
  if (st & MOE_DEV_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
  if (st & (MOE_DEV_ROUTE_RANGE | MOE_DEV_ROUTE_DUP | MOE_DEV_ROUTE_NONFINITE))
    return MOE_ERR_BAD_ROUTE;
  if (st & MOE_DEV_CAPACITY) return MOE_ERR_CAPACITY;
  if (st & MOE_DEV_BAD_SCALE) return MOE_ERR_BAD_SCALE;
  return MOE_OK;
}

moe_status moe_debug_views(moe_handle* h, moe_debug_view* v) {
  if (!h || !v) return MOE_ERR_INVALID_ARG;
  const Workspace& w = h->ws;
  v->status = w.status;
  v->counts = w.counts;
  v->offsets = w.offsets;
  v->pad_offsets = w.pad_offsets;
  v->perm = w.perm;
  v->inv = w.inv;
  v->inv_pad = w.inv_pad;
  v->a = w.a;
  v->a_sf = w.a_sf;
  v->gu = w.gu;
  v->hq = w.hq;
  v->h_sf = w.h_sf;
  v->y = w.y;
  v->rows_alloc = h->L.rows_alloc;
  v->sf_atom_bytes = kSfAtomBytes;
  v->gemm_pair = h->L.pair ? 1 : 0;
  v->gemm_ctas = gemm_grid(h);
  v->pad_rows = h->L.pad_rows;
  v->route_coop_blocks = h->sm_budget > 0 ? 0 : h->route_coop_blocks;
  return MOE_OK;
}

moe_status moe_set_profile_events(moe_handle* h, void* const* events, int32_t n) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (n == 0) {
    h->n_ev = 0;
    return MOE_OK;
  }
  if (n != 10 || !events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 10; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 10; ++i) h->ev[i] = reinterpret_cast<cudaEvent_t>(events[i]);
  h->n_ev = 10;
  return MOE_OK;
}

moe_status moe_forward_plan(moe_handle* h, int64_t num_tokens, moe_plan* out) {
  if (!h || !out || num_tokens < 0) return MOE_ERR_INVALID_ARG;
  *out = forward_plan(h, num_tokens);
  return MOE_OK;
}

moe_status moe_set_sm_budget(moe_handle* h, int32_t max_sms) {
  if (!h || max_sms < 0 || max_sms == 1) return MOE_ERR_INVALID_ARG;
  h->sm_budget = max_sms;
  return MOE_OK;
}

void moe_destroy(moe_handle* h) { delete h; }

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_CAPACITY: return "capacity exceeded";
    case MOE_ERR_NOT_BOUND: return "weights or output not bound";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_BAD_ROUTE: return "invalid routes";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MOE_ERR_BAD_SCALE: return "weight scale is not a power of two";
    case MOE_ERR_WORKSPACE: return "workspace or weight store too small";
  }
  return "unknown status";
}

}  // extern "C"
