/*
 * megamoe.h -- C ABI of the single-GPU MoE layer forward for GB300 (sm_103a).
 *
 * The layer (flashinfer PR #4069 "SM90 push FP8 mega-MoE backend",
 * Description, the forward diagram) on one GPU, where dispatch and combine
 * become a local permute and a local reduce:
 *   route + dispatch -> 1x128 FP8 E4M3 activation quantisation ->
 *   FC1 grouped GEMM (+ SwiGLU + 1x128 re-quantisation) -> FC2 grouped GEMM ->
 *   combine (top-k weighted FP32 reduction, written as BF16).
 *
 * Conventions for every call:
 *   - "d_" pointers are device pointers, "h_" pointers host pointers.  The
 *     caller allocates and owns all device memory (workspace, weight store,
 *     inputs, output); the library keeps pointers only.  The handle itself is
 *     host memory owned by the library (moe_create / moe_destroy).
 *   - BF16 tensors are passed as uint16_t bit patterns; FP8 E4M3 (OCP E4M3FN)
 *     tensors as uint8_t codes.  All arrays are dense row-major.
 *   - Streams are CUDA runtime streams (struct CUstream_st* is cudaStream_t);
 *     NULL is the legacy default stream.
 *   - Host-side argument errors return a status before anything is enqueued.
 *     Errors found on the device (bad routes, capacity, watchdog) are written
 *     to a device status word that moe_read_status returns.
 *   - No call is thread-safe on the same handle.
 */
#ifndef MEGAMOE_H
#define MEGAMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null pointer, negative size, misaligned buffer */
  MOE_ERR_UNSUPPORTED = 2,    /* dims outside the supported set (explicit, no fallback) */
  MOE_ERR_CAPACITY = 3,       /* num_tokens > max_rows, or routed rows beyond capacity */
  MOE_ERR_NOT_BOUND = 4,      /* forward before moe_bind_weights / moe_stage_inputs */
  MOE_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed */
  MOE_ERR_BAD_ROUTE = 6,      /* device: expert id out of range, duplicate, non-finite weight */
  MOE_ERR_DEVICE_TIMEOUT = 7, /* device: a bounded wait inside a kernel expired */
  MOE_ERR_BAD_SCALE = 8,      /* bind: a block scale is not a power of two in [2^-127, 2^127] */
  MOE_ERR_WORKSPACE = 9       /* workspace or weight store smaller than the query said */
} moe_status;

/* Bits of the device status word (moe_read_status). */
#define MOE_DEV_ROUTE_RANGE 0x01u     /* an expert id outside [-1, E) */
#define MOE_DEV_ROUTE_DUP 0x02u       /* the same active expert twice in one token */
#define MOE_DEV_ROUTE_NONFINITE 0x04u /* NaN/inf weight on an active route */
#define MOE_DEV_CAPACITY 0x08u        /* padded routed rows exceed the workspace capacity */
#define MOE_DEV_TIMEOUT 0x10u         /* a kernel's bounded wait expired; output undefined */
#define MOE_DEV_BAD_SCALE 0x20u       /* bind: a weight scale is not a power of two */

/* moe_dims.flags */
#define MOE_FLAG_FUSE_FC1_EPILOGUE 0x1u /* SwiGLU + 1x128 quant inside the FC1 epilogue (opt-in) */
#define MOE_FLAG_CHECK_ROUTES 0x2u      /* duplicate / finite-weight checks (range check always on) */
#define MOE_FLAG_EMIT_FC1 0x4u          /* also keep the BF16 gate||up FC1 output (debug) */
/* GEMM tactic.  MOE_FLAG_GEMM_SINGLE_CTA: one CTA per SM, expert segments
 * padded to 128 rows.  MOE_FLAG_GEMM_CTA_PAIR: CTA pairs (tcgen05
 * cta_group::2, M = 256 over two SMs), segments padded to 256 rows.  Neither:
 * chosen from expected_m -- with m = expected_m * top_k / num_experts routed
 * rows per expert, pairs when ceil(m/256)*256 < 1.13 * ceil(m/128)*128 (a
 * pair feeds its tensor cores ~13% better per row but pads more).  Buffers are
 * sized for the padding of every tactic the flags allow (256 rows unless
 * SINGLE_CTA is set), so expected_m never changes a buffer size; pass the same
 * flags to the query and to moe_create. */
#define MOE_FLAG_GEMM_SINGLE_CTA 0x8u
#define MOE_FLAG_GEMM_CTA_PAIR 0x10u
/* Test only: exercises the device watchdog.  Every kernel wait is bounded
 * (1 s); with this flag the bound is 20 ms and the first GEMM CTA withholds one
 * pipeline stage (with CTA pairs, the first pair's second CTA withholds its
 * share of one stage), so the MMA wait expires: the forward records
 * MOE_DEV_TIMEOUT, the kernel winds down (drains its copies, frees tensor
 * memory) and the context stays usable. */
#define MOE_FLAG_WATCHDOG_TEST 0x20u
/* FC1 -> FC2 in one launch.  With the fused FC1 epilogue both GEMMs can run
 * as one persistent launch (the megakernel): every FC1 tile, then every FC2
 * tile, an FC2 tile loading its hq rows once all FC1 tiles of its 128-row
 * m-tile have published them (a per-m-tile counter with a bounded wait;
 * flashinfer PR #4069, the fused FC1 -> FC2 kernel with fc1_done flags), so
 * FC2 tiles fill FC1's last wave and FC2 needs no ramp of its own.  That
 * gains about one tile round per forward and costs ~1% on long forwards, so
 * by default a forward uses one launch when its estimated tile rounds (FC1 +
 * FC2 tiles over the GEMM grid, from num_tokens, E, top_k and the tactic) are
 * at most 48, else two.  MOE_FLAG_GEMMS_ONE_LAUNCH / MOE_FLAG_SPLIT_GEMMS
 * force one or the other (not both).  Results are bit-identical either way.
 * Forwards with profiling events (moe_set_profile_events) always use two. */
#define MOE_FLAG_SPLIT_GEMMS 0x40u
#define MOE_FLAG_GEMMS_ONE_LAUNCH 0x80u
/* MXFP8 instead of the DeepSeek 1x128 / 128x128 scales: E4M3 values with one
 * power-of-two (E8M0) scale per 32 consecutive elements along K -- for the
 * activations (x and the re-quantised SwiGLU output, 1x32) and for every
 * weight row (moe_quantize_weights_mx) -- same scale rule per 32-block
 * ("32e4m3xe8m0" on flashinfer PR #4688; the SM100 MXFP8 megakernels of PR
 * #4069).  The tensor core applies every scale (one per 32-wide MMA K step),
 * so the GEMMs copy one scale atom per K block instead of one per four. */
#define MOE_FLAG_MXFP8 0x100u
/* Test only: exercises the routing kernel's grid barrier.  With this flag the
 * one-kernel routing waits at most 20 ms at its barrier, and its last block
 * withholds its arrival (forwards that route in one kernel with at least two
 * blocks, i.e. more than 512 tokens): every block records MOE_DEV_TIMEOUT and
 * marks its routes unrouted, so the forward computes no expert and writes a
 * zero output, and the context stays usable. */
#define MOE_FLAG_WATCHDOG_ROUTE_TEST 0x200u
/* Per-tensor FP8 instead of block scales: the "per_tensor" scale mode of
 * flashinfer PR #4688 (Description; the scale-mode-equalized comparison:
 * per_tensor needs offline-calibrated activation scales identical on every
 * rank, blockwise needs none).  One FP32 scale per expert weight matrix
 * (moe_quantize_weights_pt) and one static, calibrated FP32 scale per
 * activation tensor -- x and the SwiGLU output h -- given with
 * moe_set_activation_scales.  A value v with scale s is stored as
 * E4M3_RNE_sat(float(v) * float(1/s)) (saturating to +-448); the GEMMs run
 * with unit block scales and multiply their FP32 accumulators by
 * x_scale * s_w1[e] (FC1) and h_scale * s_w2[e] (FC2) before the BF16
 * rounding.  Not combinable with MOE_FLAG_MXFP8 (MOE_ERR_INVALID_ARG). */
#define MOE_FLAG_PER_TENSOR 0x400u
/* Small forwards on the single-CTA tactic run their GEMMs token-as-N
 * ("swap-AB"; flashinfer PR #4069, Limitations: no small-M swap-AB variant
 * of the fused FC1 epilogue yet; PR #4688: swap-AB token tiles chosen per
 * token bucket): when num_tokens <= 64 (so no expert has more than 64 routed
 * rows) the weights are the M = 128 operand and the first 16, 32 or 64 rows
 * of each expert segment the N operand, which leaves room for more weight
 * stages in flight and double-buffered accumulators.  Same units, same
 * arithmetic; checked against the oracle.  MOE_FLAG_NO_SWAP_AB keeps the
 * M128 x N256 kernel for every forward. */
#define MOE_FLAG_NO_SWAP_AB 0x800u
/* Opt-in: FC2 folds the combine in (flashinfer PR #4069, Description: the
 * grouped combine after FC2).  Per token and 256-column n-tile, the y chunks
 * stored so far are counted, and the warp whose count completes a token's
 * routes combines that token's columns right away -- the combine kernel's
 * arithmetic (a float fma chain over the active routes in ascending k from
 * +0, one BF16 rounding), so the output is bit-identical -- and no combine
 * kernel runs.  In the token-as-N FC2 the epilogue warps count and combine;
 * in the M128 x N256 FC2 (and the one-launch FC1 -> FC2) the epilogue warps
 * count and queue the completed (token, n-tile) pairs in shared memory for
 * two warps of their own, which combine them.  Single-CTA forwards only: ignored under CTA pairs.  Off by
 * default: it was measured slower everywhere -- 0.5-0.9% at decode T = 8 and
 * 64, 0.2% at T = 256 and 1024, 10% at the dsv2lite shape -- because each
 * completed token needs dependent L2 round trips that the combine kernel
 * overlaps across every SM, and many tokens complete only in FC2's last
 * wave. */
#define MOE_FLAG_COMBINE_IN_FC2 0x1000u

typedef struct moe_dims {
  int32_t hidden;      /* H: multiple of 128, 128..16384 */
  int32_t inter;       /* I: expert intermediate size, multiple of 128, 128..16384 */
  int32_t num_experts; /* E: 1..1024 */
  int32_t top_k;       /* K: one of 1, 2, 4, 6, 8 */
  uint32_t flags;      /* MOE_FLAG_* */
} moe_dims;

typedef struct moe_handle moe_handle;

/*
 * moe_workspace_query -- pure host arithmetic, no CUDA call.
 * Capacity contract (flashinfer PR #4069, "Contracts introduced by this PR":
 * capacity_factor bounds the GEMM, TMA and scale buffers; the query takes
 * explicit expected_m and max_rows so the tactic stays independent of the
 * memory bound).
 *   expected_m      typical tokens per forward; picks the GEMM tactic only,
 *                   never a buffer size.  >= 1.
 *   max_rows        the largest num_tokens any forward will pass.  >= 1.
 *   capacity_factor routed rows are bounded by ceil(capacity_factor *
 *                   max_rows * top_k) (plus per-expert tile padding); any
 *                   value >= 1 can never overflow.  In (0, 64].
 * Outputs (bytes): *workspace_bytes for the per-forward workspace and
 * *weight_bytes for the transformed weight store.  Any 16-byte aligned base
 * works: both sizes include slack for the library's internal 1024-byte
 * alignment of its sub-buffers.
 */
MOE_API moe_status moe_workspace_query(const moe_dims* dims, int64_t expected_m, int64_t max_rows,
                               float capacity_factor, size_t* workspace_bytes,
                               size_t* weight_bytes);

/*
 * moe_create -- the stateful layer object of flashinfer PR #4069 ("Contracts
 * introduced by this PR": a backend instance is set up once per layer with its
 * capacity and bound buffers, and forwards then only pass activations and
 * routes).  Binds dims and caller-owned device regions; creates no CUDA
 * stream and allocates no device memory.  Sets kernel attributes, so call it
 * before any stream capture.  *out receives a host handle.
 * Workspace pooling: a forward leaves nothing in the workspace that a later
 * forward reads, so several handles (the layers of a model, with equal or
 * different dims) may share one workspace of the largest size any of them
 * queried, as long as their forwards never overlap on the GPU (one stream, or
 * ordered by events).  The status word then belongs to the latest forward of
 * any of them: read it (moe_read_status) before another handle's forward.
 * The weight store and the staged output stay per handle.
 */
MOE_API moe_status moe_create(const moe_dims* dims, int64_t expected_m, int64_t max_rows,
                      float capacity_factor, void* d_workspace, size_t workspace_bytes,
                      void* d_weight_store, size_t weight_bytes, moe_handle** out);

/*
 * moe_quantize_weights -- FP32 expert weights to the format moe_bind_weights
 * takes: 128x128 blocks, scale = the smallest power of two >= amax/448 (1 for
 * an all-zero block), codes = E4M3 round-to-nearest-even of w/scale.
 *   d_w     float [num_mats, rows, cols]; rows and cols multiples of 128.
 *   d_q     uint8 [num_mats, rows, cols] (output).
 *   d_scale float [num_mats, rows/128, cols/128] (output).
 * Asynchronous on `stream`.
 */
MOE_API moe_status moe_quantize_weights(const float* d_w, int64_t num_mats, int32_t rows, int32_t cols,
                                uint8_t* d_q, float* d_scale, struct CUstream_st* stream);

/*
 * moe_quantize_weights_mx -- FP32 expert weights to the MXFP8 form that
 * moe_bind_weights takes under MOE_FLAG_MXFP8: every row quantised in 1x32
 * blocks along the columns (the K dimension of both GEMMs), scale = the
 * smallest power of two >= amax/448 (1 for an all-zero block), codes = E4M3
 * round-to-nearest-even of w/scale.
 *   d_w     float [num_mats, rows, cols]; rows and cols multiples of 128.
 *   d_q     uint8 [num_mats, rows, cols] (output).
 *   d_scale float [num_mats, rows, cols/32] (output).
 * Asynchronous on `stream`.  MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED as
 * moe_quantize_weights.
 */
MOE_API moe_status moe_quantize_weights_mx(const float* d_w, int64_t num_mats, int32_t rows,
                                           int32_t cols, uint8_t* d_q, float* d_scale,
                                           struct CUstream_st* stream);

/*
 * moe_requantize_weights_nvfp4 -- NVFP4 checkpoint weights to the format
 * moe_bind_weights takes by default (128x128 blocks, as moe_quantize_weights
 * gives): the one-time requantization through which NVFP4 checkpoints run
 * on the FP8 layer (flashinfer PR #4069, Reviewer notes).  Every value is
 *   v = e2m1(code) * e4m3(block scale) * global, rounded to float once,
 * and the 128x128 blocks of v are quantised as moe_quantize_weights does.
 *   d_codes         uint8 [num_mats, rows, cols/2]: two E2M1 codes per byte
 *                   along the columns, column 2b in the low nibble of byte b
 *                   (16-byte aligned).
 *   d_block_scales  uint8 [num_mats, rows, cols/16]: one E4M3 scale per 16
 *                   consecutive columns of a row (4-byte aligned).
 *   d_global_scales float [num_mats]: one scale per matrix.
 *   d_q, d_scale    outputs as moe_quantize_weights (d_q 16-byte aligned).
 * Block and global scales must be finite (NaN scale codes give undefined
 * output).  Asynchronous on `stream`.  MOE_ERR_INVALID_ARG for a NULL or
 * misaligned pointer or a non-positive size, MOE_ERR_UNSUPPORTED unless rows
 * and cols are multiples of 128.
 */
MOE_API moe_status moe_requantize_weights_nvfp4(const uint8_t* d_codes, const uint8_t* d_block_scales,
                                                const float* d_global_scales, int64_t num_mats,
                                                int32_t rows, int32_t cols, uint8_t* d_q,
                                                float* d_scale, struct CUstream_st* stream);

/*
 * moe_quantize_weights_pt -- FP32 expert weights to the per-tensor form that
 * moe_bind_weights takes under MOE_FLAG_PER_TENSOR: one scale per matrix,
 * s = float(amax / 448) (1 for an all-zero matrix), codes =
 * E4M3_RNE_sat(w * float(1 / s)) (the per_tensor mode of flashinfer PR #4688).
 *   d_w     float [num_mats, rows, cols]; rows and cols multiples of 128,
 *           num_mats <= 65535.
 *   d_q     uint8 [num_mats, rows, cols] (output).
 *   d_scale float [num_mats] (output; also the pass's only scratch).
 * Asynchronous on `stream`.  MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED as
 * moe_quantize_weights.
 */
MOE_API moe_status moe_quantize_weights_pt(const float* d_w, int64_t num_mats, int32_t rows,
                                           int32_t cols, uint8_t* d_q, float* d_scale,
                                           struct CUstream_st* stream);

/*
 * moe_bind_weights -- the layer holds its static weights in a transformed,
 * kernel-ready form that is built once, at set-up (flashinfer PR #4069,
 * "Contracts introduced by this PR": the stateful backend contract).  Copies
 * and transforms into the weight store (every 128x128 block of W1 and W2 one
 * contiguous 16 KB box, W1's gate and up row blocks interleaved, and the
 * scales as E8M0 plus the GEMM's scale atoms):
 *   d_w1        E4M3 [E, 2I, H]: rows [0, I) gate, rows [I, 2I) up.
 *   d_w1_scale  float [E, 2I/128, H/128], powers of two
 *               (MOE_FLAG_MXFP8: [E, 2I, H/32], one per row and 32 columns).
 *   d_w2        E4M3 [E, H, I].
 *   d_w2_scale  float [E, H/128, I/128], powers of two (MXFP8: [E, H, I/32]).
 *   Under MOE_FLAG_PER_TENSOR: d_w1_scale and d_w2_scale are float [E], one
 *   positive finite scale per expert matrix (MOE_ERR_BAD_SCALE otherwise).
 * Enqueued on `stream`, then waits for that stream: the caller may free the
 * inputs when this returns.  Returns MOE_ERR_BAD_SCALE if any scale is not a
 * power of two within the E8M0 range.
 */
MOE_API moe_status moe_bind_weights(moe_handle* h, const uint8_t* d_w1, const float* d_w1_scale,
                            const uint8_t* d_w2, const float* d_w2_scale,
                            struct CUstream_st* stream);

/*
 * moe_set_activation_scales -- the static, offline-calibrated activation
 * scales of a per-tensor layer (MOE_FLAG_PER_TENSOR; the pages' per_tensor
 * mode needs them calibrated ahead of time, identical on every rank):
 * x_scale for the layer input x, h_scale for the SwiGLU output h.  Both must
 * be positive and finite (MOE_ERR_INVALID_ARG).  MOE_ERR_UNSUPPORTED for a
 * block-scaled layer.  A per-tensor forward returns MOE_ERR_NOT_BOUND until
 * this has been called.  Enqueued on `stream` when the weights are bound
 * (the per-expert epilogue factors are computed on the device from the bound
 * weight scales), else applied by the next moe_bind_weights; may be called
 * again to change the scales, also between graph replays (the kernels read
 * them from the weight store).
 */
MOE_API moe_status moe_set_activation_scales(moe_handle* h, float x_scale, float h_scale,
                                             struct CUstream_st* stream);

/*
 * moe_stage_inputs -- binds the caller's BF16 output tensor d_out [max_rows, H]
 * ahead of the forwards that write it (flashinfer PR #4069, "Contracts
 * introduced by this PR": output binding at staging time).  May be called
 * again to rebind.
 */
MOE_API moe_status moe_stage_inputs(moe_handle* h, uint16_t* d_out);

/*
 * moe_forward -- one layer forward, asynchronous on `stream`, with no host
 * synchronisation (expert offsets stay on the device), capturable in a CUDA
 * graph.
 *   d_x         BF16 [num_tokens, H]
 *   d_topk_idx  int32 [num_tokens, K]; -1 marks a masked slot.  For graph
 *               replay with fewer live tokens, fill the tail rows with -1
 *               (flashinfer PR #6398, tail masking).
 *   d_topk_w    float [num_tokens, K]; ignored (may be NaN) on masked slots.
 *   num_tokens  0..max_rows.  0 returns MOE_OK and writes nothing.
 * Writes d_out[0:num_tokens, :] of the staged output.  Route errors set the
 * device status word; the output is then undefined.  Enqueues three to
 * eight kernels (moe_forward_plan says which): the routing as one cooperative
 * kernel (histogram, one grid-wide barrier, scan, stable scatter) when its
 * ceil(num_tokens/512) blocks can all be resident and no SM budget is set,
 * else as three kernels (histogram, scan, scatter) with the same results;
 * quant_dispatch; FC1 and FC2 as one persistent launch or two (see
 * MOE_FLAG_GEMMS_ONE_LAUNCH), with swiglu_quant between them on the unfused
 * path; combine, unless MOE_FLAG_COMBINE_IN_FC2 folds it into FC2.  The
 * status word and the forward's counters are reset first: by a memset, or by
 * the routing kernel itself when it is one block (at most 512 tokens).  Every kernel after the first is launched as a programmatic
 * dependent of the one before (it may start while its predecessor drains and
 * waits for it before touching the forward's data).
 */
MOE_API moe_status moe_forward(moe_handle* h, const uint16_t* d_x, const int32_t* d_topk_idx,
                       const float* d_topk_w, int64_t num_tokens, struct CUstream_st* stream);

/*
 * moe_read_status -- the read-back of the device-side route checker of
 * flashinfer PR #6398 ("perf(moe_ep): fuse Rubin MegaMoE forward
 * preparation", Description and the follow-up on the fused routing checker:
 * routes are validated on the device inside the forward, which stays
 * asynchronous, and the caller reads the result when it chooses).  Copies
 * the device status word of the latest forward on
 * `stream` to *h_status (MOE_DEV_* bits) and synchronises that stream: the
 * caller chooses this sync point.  Returns MOE_OK when the word is 0, else
 * the matching error (route, capacity, timeout).
 */
MOE_API moe_status moe_read_status(moe_handle* h, uint32_t* h_status, struct CUstream_st* stream);

/* moe_debug_views -- device pointers to internal buffers and their layouts,
 * for tests and tools: the debug output of flashinfer PR #4688 (the pull
 * kernel's generate_c mode keeps the raw pre-SwiGLU gate+up as BF16 so the
 * FC1 result can be checked on its own), here together with the routing
 * tables and the quantised operands.
 * The rows of a, gu, hq and y (and their scale bytes) that lie inside an
 * expert's padded segment but past its routed rows hold unspecified values:
 * the kernels compute over them but never store them or read them into a
 * routed row. */
typedef struct moe_debug_view {
  uint32_t* status;        /* device status word */
  int32_t* counts;         /* [E] rows per expert */
  int32_t* offsets;        /* [E+1] exclusive scan of counts (unpadded positions) */
  int32_t* pad_offsets;    /* [E+1] scan of counts rounded up to pad_rows (GEMM rows) */
  int32_t* perm;           /* [R] route id r = t*K + k at unpadded position pos */
  int32_t* inv;            /* [T*K] unpadded position of route r, or -1 */
  int32_t* inv_pad;        /* [T*K] padded GEMM row of route r, or -1 */
  uint8_t* a;              /* E4M3 gathered activations (padded rows), blocked: row r, column c at
                              ((r/128)*(H/128) + c/128)*16384 + (r%128)*128 + c%128 */
  uint8_t* a_sf;           /* E8M0 scale atoms of a: [rows_alloc/128][ceil(H/512)][512]
                              (MXFP8: [rows_alloc/128][H/128][512]) */
  uint16_t* gu;            /* [rows_alloc, 2I] BF16 gate||up (unfused or EMIT_FC1), else NULL */
  uint8_t* hq;             /* E4M3 re-quantised SwiGLU output, blocked like a (I columns) */
  uint8_t* h_sf;           /* E8M0 scale atoms of hq: [rows_alloc/128][ceil(I/512)][512]
                              (MXFP8: [rows_alloc/128][I/128][512]) */
  uint16_t* y;             /* [rows_alloc, H] BF16 FC2 output per padded row */
  int64_t rows_alloc;      /* padded-row capacity (multiple of 128) */
  int32_t sf_atom_bytes;   /* 512: 128 rows x 4 scale units; the scale of row r, unit
                              4q + j is byte (r%32)*16 + (r/32)*4 + j of atom q.  A unit
                              is a 128-wide K block, or a 32-wide chunk under MXFP8 */
  int32_t gemm_pair;       /* 1: GEMMs run on CTA pairs (cta_group::2), 0: one CTA per SM */
  int32_t gemm_ctas;       /* grid size of the GEMM launches */
  int32_t pad_rows;        /* rows each expert's GEMM segment is padded to */
  int32_t route_coop_blocks; /* forwards with ceil(num_tokens/512) <= this route in one cooperative
                                kernel (512 tokens per block), others in three (0: always three,
                                e.g. under an SM budget) */
} moe_debug_view;

MOE_API moe_status moe_debug_views(moe_handle* h, moe_debug_view* out);

/*
 * moe_set_profile_events -- optional per-kernel timing: when n > 0, every
 * following moe_forward records events[i] (cudaEvent_t, created by the
 * caller) before its i-th kernel and events[n-1] after the last one, on the
 * forward's stream.  Kernel order: 0 status reset, 1 route_count,
 * 2 route_scan, 3 route_scatter, 4 quant_dispatch, 5 fc1, 6 swiglu_quant
 * (skipped when fused), 7 fc2, 8 combine, 9 end.  When the routing runs as
 * one kernel, span 1 times all of it and spans 2 and 3 are empty.  n must be
 * 0 (profiling off) or 10, with every handle non-NULL.
 */
MOE_API moe_status moe_set_profile_events(moe_handle* h, void* const* events, int32_t n);

/*
 * moe_set_sm_budget -- caps the SMs the following forwards occupy, so that
 * work on another stream (a shared expert, attention of the next layer) can
 * run beside the layer (flashinfer PR #6398, the max_sm_count budget in a
 * referencing commit: capping the persistent MoE kernels lets a shared-expert
 * MLP on a side stream run at the same time).  max_sms = 0 restores the
 * default (every SM).  Otherwise 2 <= max_sms: the persistent GEMMs launch
 * min(max_sms, SM count) CTAs (one per SM; rounded down to an even count for
 * CTA pairs) and the routing keeps to its three small kernels (no
 * cooperative grid).  The short streaming kernels (quantisation, combine)
 * keep their full grids: their CTAs cannot be pinned to a subset of SMs, and
 * grids of one CTA per budgeted SM made the dsv2lite-shaped layer 25% slower
 * at a 144-SM budget (3% with full grids).  Results
 * are bit-identical for every budget.  Errors: MOE_ERR_INVALID_ARG for a NULL
 * handle or max_sms < 0 or == 1.
 */
MOE_API moe_status moe_set_sm_budget(moe_handle* h, int32_t max_sms);

/*
 * moe_forward_plan -- the kernels moe_forward enqueues for num_tokens tokens
 * with the handle's current flags and SM budget, without profiling events
 * (the routing form, one or two GEMM launches: see MOE_FLAG_GEMMS_ONE_LAUNCH).
 * Pure host arithmetic, no CUDA call; the same function the forward uses.
 * num_tokens 0 gives all zeros.  MOE_ERR_INVALID_ARG for a NULL argument or
 * num_tokens < 0.
 */
typedef struct moe_plan {
  int32_t route_kernels;  /* 1 (one cooperative kernel) or 3 */
  int32_t gemm_launches;  /* 1 (FC1 -> FC2 in one persistent launch) or 2 */
  int32_t swiglu_kernels; /* 1 on the unfused path, else 0 */
  int32_t kernels;        /* all of them: + quant_dispatch (+ combine unless folded) */
  int32_t swap_ab_tokens; /* token tile of the token-as-N GEMMs (16, 32, 64), or 0 */
  int32_t combine_in_fc2; /* 1: the combine is folded into FC2 (MOE_FLAG_COMBINE_IN_FC2; no combine kernel) */
} moe_plan;

MOE_API moe_status moe_forward_plan(moe_handle* h, int64_t num_tokens, moe_plan* out);

/*
 * moe_route_noalloc -- the routing step alone, allocating nothing.  The pages
 * have no counterpart to this call; it exists for callers that cannot
 * allocate device memory and have no workspace to offer, for example a plugin
 * run from inside another runtime's enqueue callback, where cudaMalloc would
 * synchronise the device and is not allowed, or code that must not grow the
 * host framework's memory pool.
 *
 * Computes what moe_forward's routing kernels compute, into the caller's
 * buffers: route validation (bits OR-ed into *d_status, which this call first
 * clears), per-expert counts d_counts [E], the exclusive scan d_offsets
 * [E+1], and the stable permutation d_perm [num_tokens*top_k] (first
 * offsets[E] entries meaningful) with its inverse d_inv [num_tokens*top_k]
 * (-1 for masked slots).  Inputs as for moe_forward.  check_routes != 0 adds
 * the duplicate and finite-weight checks.
 *
 * Scratch: a fixed file-scope device array of about 0.9 MiB, present in every
 * CUDA context that loads the library until that context is destroyed (for
 * the runtime's primary context: until the process exits).  Limits:
 * num_tokens * top_k <= 131072, ceil(num_tokens / 128) * num_experts <= 32768,
 * num_experts <= 1024; larger inputs return MOE_ERR_CAPACITY before anything
 * is enqueued.  The array's device address belongs to one context: the first
 * call made in a context (the one current on the calling thread, primary or a
 * context the caller made current) looks it up (cudaGetSymbolAddress) and
 * caches it under the context's unique id, so make that first call before
 * any stream capture.  Every call in a context uses the same array, so calls
 * that overlap on the GPU (other streams, other threads) race and corrupt
 * each other's results: order them on one stream.  The array keeps the last
 * call's contents; nothing in it needs to start at zero.
 * Errors: MOE_ERR_UNSUPPORTED for top_k or num_experts outside the set above;
 * MOE_ERR_INVALID_ARG for num_tokens < 0 or a NULL pointer (d_topk_idx,
 * d_topk_w, d_perm and d_inv may be NULL when num_tokens == 0);
 * MOE_ERR_CAPACITY as above; MOE_ERR_CUDA when a CUDA call fails.
 * num_tokens == 0 clears *d_status, zeroes d_counts and d_offsets and writes
 * nothing else.  Asynchronous on stream.
 */
MOE_API moe_status moe_route_noalloc(const int32_t* d_topk_idx, const float* d_topk_w,
                                     int64_t num_tokens, int32_t top_k, int32_t num_experts,
                                     int32_t check_routes, int32_t* d_counts, int32_t* d_offsets,
                                     int32_t* d_perm, int32_t* d_inv, uint32_t* d_status,
                                     struct CUstream_st* stream);

/* moe_destroy -- frees the host handle (lifecycle only; the pages have no
 * passage on it).  Device memory stays the caller's.  NULL is a no-op. */
MOE_API void moe_destroy(moe_handle* h);
/* moe_status_str -- a static text for a status code (error reporting only;
 * the pages have no passage on it). */
MOE_API const char* moe_status_str(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MEGAMOE_H */
