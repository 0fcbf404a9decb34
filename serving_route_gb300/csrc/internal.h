// internal.h -- host-side layout of the workspace / weight store and the
// launchers each kernel file exports to the C-ABI layer (api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/megamoe.h"

namespace mm {

// Device buffers carved out of the caller's workspace (all 1024-byte aligned).
struct Workspace {
  uint32_t* status;        // device status word (MOE_DEV_* bits)
  int32_t* total_mtiles;   // number of 128-row GEMM tiles of this forward
  uint32_t* grid_sync;     // arrival counter of the one-kernel routing (zeroed before each forward)
  int32_t* gemm_sched;     // [2] unit counters of the FC1 and FC2 launches (zeroed before each forward)
  int32_t* cmb_cnt;        // [max_rows][ceil(H/256)] stored y chunks per token and n-tile (zeroed
                           // before each forward that folds the combine into FC2)
  int32_t* fc1_done;       // [max_mtiles] FC1 tiles published per m-tile (zeroed before each forward)
  int32_t* counts;         // [E]
  int32_t* offsets;        // [E+1]
  int32_t* pad_offsets;    // [E+1]
  int32_t* mtile_expert;   // [max_mtiles]
  int32_t* block_counts;   // [nb_max][E] routes per (128-token block, expert)
  int32_t* base_u;         // [nb_max][E] unpadded start of a block's expert run
  int32_t* base_p;         // [nb_max][E] padded start of a block's expert run
  int32_t* perm;           // [max_rows*K]
  int32_t* inv;            // [max_rows*K]
  int32_t* inv_pad;        // [max_rows*K]
  uint8_t* a;              // blocked [rows_alloc/128][H/128][128][128]
  uint8_t* a_sf;           // atoms [rows_alloc/128][ceil(H/512)][512]
  uint16_t* gu;            // [rows_alloc, 2I] or nullptr
  uint8_t* hq;             // blocked [rows_alloc/128][I/128][128][128]
  uint8_t* h_sf;           // atoms [rows_alloc/128][ceil(I/512)][512]
  uint16_t* y;             // [rows_alloc, H]
};

struct WeightStore {
  uint8_t* w1;     // [E][2I/128][H/128][128][128]: 128x128 blocks, each contiguous; row blocks
                   // in the order gate 0, up 0, gate 1, up 1, ... (one 256-row FC1 tile = gate j + up j)
  uint8_t* w2;     // [E][H/128][I/128][128][128]
  uint8_t* w1_sf;  // [E, 2I/128, H/128] E8M0, in the interleaved row-block order of w1
  uint8_t* w2_sf;  // [E, H/128, I/128] E8M0
  uint8_t* w1_sfatoms;  // [E][2I/128][ceil(H/512)][512]: w1_sf as GEMM scale atoms
  uint8_t* w2_sfatoms;  // [E][H/128][ceil(I/512)][512]
  // per-tensor format: float [4E + 2] = the weight scales s_w1[E], s_w2[E],
  // the epilogue factors x_scale * s_w1[E], h_scale * s_w2[E], then the
  // reciprocals 1/x_scale, 1/h_scale (nullptr in the block-scaled formats)
  float* pt;
};

struct Layout {
  int H, I, E, K;
  bool mx;             // MXFP8: one scale per 32-wide K chunk (else 1x128 / 128x128)
  bool pt;             // per-tensor scales (block scales all 1; factors in the epilogues)
  int pad_rows;        // expert segments padded to this many rows (128, or 256 for CTA pairs)
  bool pair;           // GEMMs run on CTA pairs (tcgen05 cta_group::2)
  int64_t max_rows;
  int64_t cap_rows;    // routed-row capacity before padding
  int64_t rows_alloc;  // padded GEMM rows (multiple of 128)
  int64_t nb_max;      // 128-token blocks of max_rows
  bool keep_gu;
  size_t ws_bytes, w_bytes;
  // byte offsets inside the workspace / weight store
  size_t o_fc1_done;   // [max_mtiles] int32 counters of the megakernel, right after the status
  size_t o_cmb;        // [max_rows][ceil(H/256)] int32 counters of the folded combine, after those
  size_t o_status, o_counts, o_offsets, o_pad_offsets, o_mtile_expert, o_block_counts, o_base_u,
      o_base_p, o_perm, o_inv, o_inv_pad, o_a, o_a_sf, o_gu, o_hq, o_h_sf, o_y;
  size_t o_w1, o_w2, o_w1_sf, o_w2_sf, o_w1_sfatoms, o_w2_sfatoms, o_pt;
};

// Scale atoms along K: one per four 128-wide K blocks (one byte per block),
// or under MXFP8 one per K block (one byte per 32-wide chunk).
inline int64_t atoms_along_k(int64_t kblocks, bool mx) { return mx ? kblocks : (kblocks + 3) >> 2; }

// layout.cpp-style pure host arithmetic (api.cu)
moe_status compute_layout(const moe_dims* d, int64_t expected_m, int64_t max_rows,
                          float capacity_factor, Layout* L);

// route.cu
// One cooperative kernel (count, grid barrier, scan, scatter) when its
// ceil(T/512) blocks can all be resident (coop_max_blocks: the device's limit
// for the fused kernel, 0 = never) and ws.grid_sync is zero; otherwise the
// three kernels route_count / route_scan / route_scatter.  Same outputs.
// watchdog_test: the one-kernel form's last block withholds its arrival at
// the grid barrier, whose bound drops to 20 ms (test only).
// zero_words: when the one-kernel form runs as a single block (T <= 512),
// it clears that many 32-bit words from ws.status on (the forward's status
// word and counters) before anything else; the caller then skips its memset.
cudaError_t launch_route(const Workspace& ws, const Layout& L, const int32_t* topk_idx,
                         const float* topk_w, int64_t T, bool check, cudaStream_t s,
                         cudaEvent_t const* ev, int coop_max_blocks, bool watchdog_test = false,
                         int64_t zero_words = 0);
// Largest grid of the one-kernel routing that is co-resident on the current
// device for E experts (0 if cooperative launch is unavailable).
int route_fused_max_blocks(int E);

// quant.cu
// Resident blocks (all SMs) of quant_dispatch with two or four units per
// warp pass (batch 2 or 4) for format fmt (0 1x128, 1 MXFP8, 2 per-tensor);
// 0 if the query fails.
int quant_dispatch_resident(int fmt, int batch);
// pdl: launch as a programmatic dependent of the previous kernel on `s`;
// max_ctas: grid cap of the streaming kernels; resident2 / resident4: the
// two forms' resident blocks (four units per warp where that makes one wave)
// pt_rx / pt_rh: the per-tensor reciprocals in the weight store (per-tensor only)
cudaError_t launch_quant_dispatch(const Workspace& ws, const Layout& L, const uint16_t* x,
                                  int64_t T, cudaStream_t s, bool pdl, int max_ctas,
                                  int resident2, int resident4, const float* pt_rx);
cudaError_t launch_swiglu_quant(const Workspace& ws, const Layout& L, int max_ctas, cudaStream_t s,
                                bool pdl, const float* pt_rh);
cudaError_t launch_quantize_weights_pt(const float* w, int64_t nmat, int rows, int cols, uint8_t* q,
                                       float* scale, cudaStream_t s);
cudaError_t launch_pt_set_scales(const WeightStore& wst, const Layout& L, float x_scale,
                                 float h_scale, cudaStream_t s);
cudaError_t launch_quantize_weights(const float* w, int64_t nmat, int rows, int cols, uint8_t* q,
                                    float* scale, cudaStream_t s);
// NVFP4 checkpoint weights (codes [nmat, rows, cols/2], E4M3 scales
// [nmat, rows, cols/16], float global [nmat]) -> the 128x128 FP8 format.
cudaError_t launch_requant_nvfp4(const uint8_t* codes, const uint8_t* sblk, const float* gs,
                                 int64_t nmat, int rows, int cols, uint8_t* q, float* scale,
                                 cudaStream_t s);
cudaError_t launch_quantize_weights_mx(const float* w, int64_t nmat, int rows, int cols, uint8_t* q,
                                       float* scale, cudaStream_t s);
cudaError_t launch_bind_transform(const WeightStore& wst, const Layout& L, const uint8_t* w1,
                                  const float* w1s, const uint8_t* w2, const float* w2s,
                                  uint32_t* status, cudaStream_t s);

// gemm.cu
// kModeMega: one persistent launch of both GEMMs -- every FC1 tile (fused
// epilogue; gate||up also stored when that phase's `out` is set), then every
// FC2 tile, each FC2 tile's loads waiting for its m-tile's fc1_done count.
enum GemmMode { kModeY = 0, kModeGU = 1, kModeFused = 2, kModeFusedGU = 3, kModeMega = 4 };
struct GemmArgs {
  const uint8_t* sfa;          // scale atoms of A: [mblocks][KQ][512]
  const uint8_t* sfb;          // scale atoms of B: [E][NB][KQ][512]
  const int32_t* mtile_expert;
  const int32_t* total_mtiles;
  // routed rows and padded segment start per expert: an m-tile's rows past
  // pad_offsets[e] + counts[e] are padding that nothing downstream reads
  const int32_t* counts;
  const int32_t* pad_offsets;
  int KB;                      // K / 128
  int KQ;                      // scale atoms along K (atoms_along_k)
  int mx;                      // MXFP8: an atom per K block, MMA k uses byte k
  int NT;                      // 256-wide N tiles per expert
  int N;                       // B rows per expert
  int NB;                      // N / 128
  int max_mtiles;
  uint16_t* out;               // kModeY: y; kModeGU/kModeFusedGU: gu
  int64_t ld_out;              // elements per output row
  int inter;                   // I: column offset of the up half in gu
  uint8_t* hq;                 // fused: blocked [rows/128][I/128][128][128]
  uint8_t* h_sf;               // fused: scale atoms [mblocks][I/128][512]
  int IB;                      // I / 128
  uint32_t* status;
  uint64_t wait_limit_ns;      // bound of every mbarrier wait (1 s; 20 ms in the watchdog test)
  int watchdog_test;           // 1: CTA 0 withholds one stage so its MMA wait expires
  // kModeMega: per 128-row m-tile, the FC1 tiles whose fused-epilogue stores
  // are complete and visible (zeroed before each forward); FC2 tiles of an
  // m-tile start loading when it reaches fc1_ntiles
  int32_t* fc1_done;
  int fc1_ntiles;
  // single-CTA launches: the dynamic schedule's unit counter (zeroed before
  // each forward; one per launch), or nullptr for the static order
  int32_t* sched;
  // per-tensor format: per-expert factors applied to the FP32 accumulator
  // before the BF16 rounding, and (FC1) the h scale's float reciprocal;
  // nullptr in the block-scaled formats
  const float* pt_scale;
  const float* pt_rh;
  // FC2 with the combine folded in (nullptr cmb_cnt: the combine kernel runs
  // after): per token and 256-column n-tile, the stored y chunks (token-as-N:
  // one count per route and lane-quadrant warp; M128 x N256: one per route
  // and column half; zeroed before each forward); the warp that completes a
  // token's count combines that column range of the token into the BF16
  // output, as the combine kernel does
  int32_t* cmb_cnt;         // [T][NT]
  uint16_t* cmb_out;        // BF16 [T, H]
  const float* cmb_w;       // top-k weights [T, K]
  const int32_t* cmb_inv;   // padded GEMM row of route t*K + k, or -1
  const int32_t* cmb_perm;  // route id at each unpadded sorted position
  const int32_t* cmb_offsets;  // unpadded segment starts [E+1]
  int cmb_T, cmb_K;
};
cudaError_t gemm_set_attributes();
int gemm_max_pairs();
// tmB: the blocked weight store as a 3-D map (one 128x128 block per box).
// pair: CTA-pair kernel (tmSfa / tmSfb = the A / B
// scale atoms as 2-D uint32 tensors of 512-byte rows); otherwise the
// single-CTA kernel (scale atoms by bulk copy from
// g.sfa / g.sfb).  tmY: the FC2 output [rows, H] BF16 with
// 32x32 boxes and 64-byte swizzle (TMA stores of kModeY).  ctas: grid size
// (even for pairs).
cudaError_t launch_gemm(GemmMode mode, bool pair, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        const CUtensorMap* tmSfa, const CUtensorMap* tmSfb, const CUtensorMap* tmY,
                        const GemmArgs& g, int ctas, cudaStream_t s, bool pdl);
// Both GEMMs in one launch (kModeMega): phase 0 = FC1 with tmA/tmB/tmSfa/tmSfb
// and g (fused epilogue), phase 1 = FC2 with tmA2/tmB2/tmSfa2/tmSfb2, tmY and
// g2 (g2.fc1_done / fc1_ntiles set).
cudaError_t launch_gemm_mega(bool pair, const CUtensorMap* tmA, const CUtensorMap* tmB,
                             const CUtensorMap* tmSfa, const CUtensorMap* tmSfb,
                             const CUtensorMap* tmA2, const CUtensorMap* tmB2,
                             const CUtensorMap* tmSfa2, const CUtensorMap* tmSfb2,
                             const CUtensorMap* tmY, const GemmArgs& g, const GemmArgs& g2, int ctas,
                             cudaStream_t s, bool pdl);

// gemm_swap.cu: the token-as-N form of the same units for forwards that
// route at most ntok (16, 32 or 64) rows to any expert.  tmX / tmX2: the
// activation buffers (A, hq) as blocked maps whose box is ntok rows high;
// tmW / tmW2: the weight maps of launch_gemm.  Scale atoms by bulk copy from
// g.sfa / g.sfb.  kModeMega takes both phases (g2.fc1_done set).
cudaError_t gemm_swap_set_attributes();
cudaError_t launch_gemm_swap(GemmMode mode, int ntok, const CUtensorMap* tmX, const CUtensorMap* tmW,
                             const CUtensorMap* tmX2, const CUtensorMap* tmW2, const GemmArgs& g,
                             const GemmArgs& g2, int ctas, cudaStream_t s, bool pdl);

// combine.cu
cudaError_t launch_combine(const Workspace& ws, const Layout& L, const float* topk_w,
                           uint16_t* out, int64_t T, cudaStream_t s, bool pdl, int max_ctas);

}  // namespace mm
