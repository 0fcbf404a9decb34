// common.cuh -- device helpers of the MoE layer kernels (sm_103a only).
//
// Inline PTX wrappers for mbarriers, TMA, and the 5th-generation tensor core
// (tcgen05: TMEM allocation, block-scaled MMA, shared->TMEM copies, TMEM
// loads), plus the number-format helpers every kernel shares: the power-of-two
// 1x128 scale rule, E4M3 packing through the hardware convert, the E8M0 scale
// atom layout, and SwiGLU.
#pragma once

#include <cuda.h>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/megamoe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "this library is written for sm_103a only"
#endif

namespace mm {

// ----------------------------------------------------------------------------
// Scale atoms: the E8M0 scale bytes of 128 rows x 4 consecutive 128-wide K
// blocks, 512 bytes, in the order the block-scaled MMA reads them from TMEM
// after a 32x128b.warpx4 copy: row r of the 128-row tile sits at byte
// (r % 32) * 16 + (r / 32) * 4 + j, where j is the K block within the group of
// four.  A 1x128 (or 128x128) scale covers all four 32-wide K chunks of its
// block, so the four MMAs of K block 4q + j all select byte j through the
// scale-factor ids of the instruction descriptor, and one copy into TMEM
// serves four K blocks.
// ----------------------------------------------------------------------------
constexpr int kSfAtomBytes = 512;

__host__ __device__ __forceinline__ int64_t sf_kgroups(int64_t kblocks) { return (kblocks + 3) >> 2; }

__host__ __device__ __forceinline__ int64_t sf_atom_offset(int64_t row, int64_t kblock,
                                                          int64_t kblocks) {
  return ((row >> 7) * sf_kgroups(kblocks) + (kblock >> 2)) * kSfAtomBytes + (row & 31) * 16 +
         ((row & 127) >> 5) * 4 + (kblock & 3);
}

// Byte offset of (row, column) in a blocked E4M3 activation buffer: every
// 128-row x 128-column block is one contiguous 16 KB box,
// [rows / 128][cols / 128][128][128], so a GEMM stage's A box is one
// sequential read.
__host__ __device__ __forceinline__ int64_t blocked_offset(int64_t row, int64_t col, int64_t cols) {
  return (((row >> 7) * (cols >> 7) + (col >> 7)) << 14) + ((row & 127) << 7) + (col & 127);
}

// Smallest e with amax <= 448 * 2^e, kept in [-127, 127]; amax == 0 gives 0.
// amax = m * 2^E, m in [1, 2): e = E - 8 when m <= 1.75, else E - 7
// (448 = 1.75 * 2^8).  Subnormal amax lies below every kept scale.
__device__ __forceinline__ int pow2_scale_exp(float amax) {
  uint32_t b = __float_as_uint(amax);
  if (b == 0u) return 0;
  uint32_t ef = b >> 23;
  if (ef == 0u) return -127;
  int e = (int)ef - 127 - 8 + (((b & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as a float, exact for e in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2_neg(int e) {
  int k = -e;
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

// Two floats to two E4M3 codes (round to nearest even, saturating), low byte = a.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  __nv_fp8x2_storage_t v = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)v;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// SwiGLU of one gate/up pair: silu(g) * u = g / (1 + exp(-g)) * u, in float,
// with the hardware exponential and approximate divide (a few ulp of float,
// far below the BF16 rounding of the gate/up inputs).  For g < -88 the
// exponential overflows and the quotient is 0, the limit of silu.  The fused
// FC1 epilogue and the unfused kernel both call this one function, so they
// agree bit for bit.
__device__ __forceinline__ float swiglu(float g, float u) {
  const float s = __fdividef(g, __fadd_rn(1.0f, __expf(-g)));
  return __fmul_rn(s, u);
}

// Profiling events are recorded as external event nodes when the stream is
// being captured, so per-kernel timing also works inside CUDA graphs.
static inline void record_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

// 32-byte global store (one full sector); dst must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* dst, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t a4, uint32_t a5, uint32_t a6,
                                             uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

__device__ __forceinline__ void record_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// ----------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of a forward after the first is
// launched with programmatic stream serialisation: it may start while its
// predecessor finishes, and executes pdl_wait() before it touches global
// memory that any earlier kernel of the forward writes or reads (the wait
// returns once the predecessor grid has completed and its writes are
// visible; completion is transitive along the chain).  pdl_trigger() lets the
// successor launch once every CTA of this grid has issued it or exited.  A
// kernel that is itself a dependent issues pdl_trigger() only after its
// pdl_wait(): quant_dispatch triggering at its very start (so that the GEMM
// after it could launch while the routing still ran) read routing tables the
// routing had not yet written (a one-token forward's A row came out wrong).
// ----------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#ifndef __CUDACC_RTC__
// Launch `kernel` on `s`; when `pdl`, with programmatic stream serialisation
// (plus up to one extra attribute, e.g. a cluster shape).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, bool pdl, const cudaLaunchAttribute* extra,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (extra) attr[n++] = *extra;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#endif

// ----------------------------------------------------------------------------
// Shared memory, mbarriers, TMA.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

// try_wait with acquire at cluster scope: pairs with release.cluster arrives
// from the other CTA of a pair (its shared-memory writes become visible).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every wait in these kernels is bounded: after `limit_ns` (or once another
// role of the CTA has given up, *abort != 0) it records MOE_DEV_TIMEOUT and
// returns false so the kernel can wind down instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, uint32_t* status,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  auto try_once = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (try_once()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (try_once()) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      record_status(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// Non-blocking probes of a phase: the fast path of every wait below.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

// The bounded wait kept out of line: inlined into the MMA issue loop, the
// polling loop slows that loop even when it is never entered.
template <bool CLUSTER>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort,
                                            uint32_t* status, uint64_t limit_ns) {
  return mbar_wait_bounded<CLUSTER>(bar, parity, abort, status, limit_ns);
}

// Bounded wait: one non-blocking probe, then the out-of-line polling loop.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, uint64_t limit_ns = kWaitLimitNs) {
  const bool done = CLUSTER ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity);
  return done || mbar_wait_slow<CLUSTER>(bar, parity, abort, status, limit_ns);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy global accesses with its async-proxy
// (TMA / bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Loads with acquire semantics at GPU scope (counters other CTAs publish).
__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int32_t ld_acquire_gpu_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Relaxed (strong) load at GPU scope; a later fence_acq_rel_gpu() turns a
// value it read from a release into an acquire.
__device__ __forceinline__ int32_t ld_relaxed_gpu_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Atomic add with release semantics at GPU scope: everything this thread's
// CTA made visible to it before is visible to a thread that acquires the sum.
__device__ __forceinline__ void red_release_gpu_add(int32_t* p, int32_t v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// 2-D tiled TMA load (box given by the tensor map) into shared memory,
// completing `bytes` of transaction on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint32_t bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// 2-D TMA store of one box from shared memory, tracked as a bulk async-group.
__device__ __forceinline__ void tma_store_2d(const void* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   (uint64_t)map),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store of this thread has read its source.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"((uint64_t)src), "r"(bytes), "r"(bar)
      : "memory");
}

// ----------------------------------------------------------------------------
// Thread-block clusters (the CTA pair of the 2-SM GEMM).
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// All threads of all CTAs of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar_cluster, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
                   bar_cluster),
               "r"(bytes)
               : "memory");
}

// Arrive on a barrier of either CTA of the pair with no memory ordering: for
// signals that carry no data through memory (an accumulator whose TMEM reads
// have already completed), where a cluster-scope release would wait for the
// thread's outstanding global stores.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// 2-D TMA load into this CTA's shared memory that completes its bytes on an
// mbarrier of either CTA of the pair (the leader's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* map, uint32_t bar_cluster,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

// 3-D tiled TMA loads (the blocked weight store: {128 bytes, rows, row block}).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint32_t bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* map, uint32_t bar_cluster,
                                                 int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, accumulators in tensor memory).
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// CTA-pair forms: one warp in each CTA of the pair runs alloc / relinquish /
// dealloc together; the same columns are reserved in both SMs' TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Pair forms: completion of this thread's prior cta_group::2 operations,
// arriving on the barrier at the same offset in every CTA of `mask`.
__device__ __forceinline__ void tc_commit_pair_multicast(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Shared-memory matrix descriptor, K-major operand staged by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29,
// unused for swizzled K-major), stride byte offset >> 4 (32-45), descriptor
// version 1 (bit 46), swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Descriptor of a 512-byte scale atom (32 rows x 16 bytes, no swizzle, 8-row
// core matrices 128 bytes apart) for the 32x128b shared->TMEM copy.
__device__ __forceinline__ uint64_t sdesc_sf_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128u >> 4) << 16;
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4 with block scales:
// A and B E4M3 (format 0, bits 7-9 / 10-12), both K-major (bits 15, 16 = 0),
// N >> 3 (bits 17-22), scale type E8M0 (bit 23), M >> 7 (bits 27-28), and the
// scale-factor ids (the byte of each 32-bit TMEM scale word the MMA uses):
// bits 4-5 for B, 29-30 for A.
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(int M, int N, uint32_t sf_id = 0) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 7) << 27) | (sf_id << 4) |
         (sf_id << 29);
}

// D[tmem] (+)= (A * 2^sfa) x (B * 2^sfb)^T, FP32 accumulation, K = 32.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// CTA-pair MMA: M = 256 rows, 128 from each CTA's shared memory into its own
// TMEM; B split by rows between the two CTAs; issued by the leader CTA.
__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t sfa_tmem,
                                                 uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Pair form of the scale-atom copy: each CTA's atom (same offset) to its TMEM.
__device__ __forceinline__ void tc_cp_sf_atom_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Shared -> TMEM copy of one scale atom: 32 lanes x 128 bits, replicated to
// the four 32-lane quadrants.
__device__ __forceinline__ void tc_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace mm
