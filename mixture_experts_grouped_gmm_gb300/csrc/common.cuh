// Shared device helpers for the sm_103a kernels: args-block accessors,
// mbarrier / TMA / tcgen05 inline PTX, bounded waits, e4m3 conversion.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mgemm.h"

namespace mgemm {

// ---------------------------------------------------------------- host errors
// Records a failed CUDA call for mgemm_last_error() (per thread) and maps it
// to MGEMM_ECUDA.
void note_error(const char *where, int code);
inline int cuda_rc(cudaError_t e, const char *where) {
  if (e == cudaSuccess) return MGEMM_OK;
  note_error(where, (int)e);
  return MGEMM_ECUDA;
}

// Tiled tensor map with 128-byte swizzle (or none) and zero fill outside the
// tensor (dims[0] contiguous; strides in bytes for dims 1..rank-1).
bool make_tensor_map(CUtensorMap *m, bool byte_elems, int rank, const void *base, const uint64_t *dims,
                     const uint64_t *strides, const uint32_t *box, bool swizzle128 = true);
// cuTensorMapEncodeTiled needs a current context; a thread that has made no
// CUDA call yet (an autograd worker, say) has none.  Makes the current
// device's primary context current, once per thread.
int ensure_context();
// Number of SMs of the current device (cached per device), or < 0 on error.
int sm_count_cached();

// Launch with programmatic stream serialization: the kernel's CTAs may be
// placed while the previous kernel of the stream is still finishing, which
// hides the launch latency between the two.  Every kernel launched this way
// calls pdl_wait() before it reads or writes global memory (the wait ends when
// the previous grid has completed and its writes are visible, so the ordering
// is that of a plain launch) and pdl_trigger() only after that wait: the next
// launch can then start only once every CTA of this one is resident, so it
// never holds an SM that a CTA of this grid still needs.  cluster_x > 1 also
// launches clusters of that many CTAs.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, unsigned cluster_x,
               const char *what, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cuda_rc(cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...), what);
}

// ---------------------------------------------------------------- args block
// Rows of each group in the padded column-major FP8 layout are rounded up to this.
constexpr int kColPad = MGEMM_COL_PAD;
static_assert(kColPad % 16 == 0, "padded groups keep 16-byte alignment");

struct ArgsLayout {
  size_t offsets, active, mtile_start, wgrad_order, poffsets, ptile_start, bytes;
};

__host__ __device__ constexpr ArgsLayout args_layout(int E) {
  ArgsLayout L{};
  L.offsets = 24;
  L.active = L.offsets + 8 * (size_t)(E + 1);
  L.mtile_start = L.active + 4 * (size_t)E;
  L.wgrad_order = L.mtile_start + 4 * (size_t)(E + 1);
  L.poffsets = (L.wgrad_order + 4 * (size_t)E + 7) & ~(size_t)7;
  L.ptile_start = L.poffsets + 8 * (size_t)(E + 1);
  L.bytes = (L.ptile_start + 4 * (size_t)(E + 1) + 15) & ~(size_t)15;
  return L;
}

struct ArgsView {
  int *status;
  int *work;  // header word 3: work counter, 0 between launches
  const int *n_active;
  const int64_t *offsets;
  const int *active;
  const int *mtile_start;
  const int *wgrad_order;
  const int64_t *poffsets;  // padded column-major layout: group e starts at poffsets[e]
  const int *ptile_start;   // prefix over active groups of ceil(m / 256): row-tile pairs of CTA pairs
  __device__ ArgsView(const void *base, int E) {
    uint8_t *b = (uint8_t *)base;
    ArgsLayout L = args_layout(E);
    status = (int *)b;
    work = (int *)(b + 12);
    n_active = (const int *)(b + 4);
    offsets = (const int64_t *)(b + L.offsets);
    active = (const int *)(b + L.active);
    mtile_start = (const int *)(b + L.mtile_start);
    wgrad_order = (const int *)(b + L.wgrad_order);
    poffsets = (const int64_t *)(b + L.poffsets);
    ptile_start = (const int *)(b + L.ptile_start);
  }
};

// Records the first device-side error; later ones do not overwrite it.
__device__ __forceinline__ void set_status(int *status, int code) { atomicCAS(status, 0, code); }

// Programmatic dependent launch (see launch_pdl): wait for the previous grid
// of the stream (a no-op for a plain launch), then let the next one be placed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- PTX: basics
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up (returns
// false) after kWaitLimitNs of wall time or when *abort_flag becomes non-zero,
// so no kernel of this library can spin forever.  A build with
// MGEMM_WAIT_LIMIT_NS=0 (used only to test the give-up path) makes every
// pipeline wait a single non-blocking test: a phase that is not already
// complete counts as a timeout.
#ifndef MGEMM_WAIT_LIMIT_NS
#define MGEMM_WAIT_LIMIT_NS 1000000000ull  // 1 s
#endif
constexpr uint64_t kWaitLimitNs = MGEMM_WAIT_LIMIT_NS;
// The drain after a give-up (copies and MMAs already issued must land before
// shared and tensor memory are released) always waits up to 1 s: those
// operations complete on their own within microseconds.
constexpr uint64_t kDrainLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity, const volatile int *abort_flag,
                                              uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 255u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const volatile int *abort_flag) {
  if constexpr (kWaitLimitNs == 0) return mbar_test_wait(smem_u32(bar), parity);
  return mbar_wait_for(bar, parity, abort_flag, kWaitLimitNs);
}

// The drain's wait (see kDrainLimitNs); false if it gave up.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, nullptr, kDrainLimitNs);
}

// mbar_wait for a whole converged warp: every lane waits, and all lanes get
// the same answer (a timeout seen by any lane counts for the warp), so the
// code after it never diverges into warp-collective instructions.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, const volatile int *abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// mbar_wait_warp with acquire at cluster scope: the arrivals come from the
// other CTA of the pair (released at cluster scope) and order its writes
// into this CTA's shared memory before the reads that follow.
__device__ __forceinline__ bool mbar_wait_cluster_warp(uint64_t *bar, uint32_t parity, const volatile int *abort_flag) {
  const uint32_t a = smem_u32(bar);
  auto test = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    return ok != 0;
  };
  bool ok = test();
  if (!ok) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
      if (test()) {
        ok = true;
        break;
      }
      if ((i & 255u) == 0 && ((abort_flag && *abort_flag) || global_timer_ns() - t0 > kWaitLimitNs)) break;
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// 16 bytes global -> shared, asynchronous (src_bytes 0: zeros, nothing read);
// cp_async_mbar_arrive makes an mbarrier arrival once this thread's earlier
// copies have landed (the barrier's count includes that arrival).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Shared -> global tiled store (bulk-group completion).
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1,
                                            int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, const void *src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all of this thread's bulk groups have completed (writes visible).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]; 16-bit inputs, fp32 accumulator.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same for 8-bit float inputs (e4m3 here).
// Block-scaled e4m3 MMA (one ue8m0 scale per 32 contraction elements of each
// row of A and B, read from tensor memory at sfa / sfb).
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// Shared memory -> tensor memory copy of scale factors: 32 rows of 16 bytes
// to lanes 0-31 of each lane quarter (4 columns).
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// ---------------------------------------------------------------- CTA pairs
// A cluster of two CTAs sharing one tensor-core operation (tcgen05 with
// cta_group::2): the even-ranked CTA issues the MMA, whose A operand is the
// two CTAs' 128-row halves and whose B operand is the two CTAs' N/2-column
// halves (same shared-memory offsets in both), and whose accumulator is the
// two CTAs' TMEM (128 lanes each).  Every tcgen05 instruction of such a
// kernel carries cta_group::2.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t ncluster_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// The shared::cluster address of `p` (a shared variable of this CTA) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// Store a 32-bit value into shared memory of another CTA of the cluster.
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr_, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr_), "r"(v) : "memory");
}
// Every thread of both CTAs (all warps, converged).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of the pair's leader CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *m, uint32_t cluster_bar, int c0,
                                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(cluster_bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *m, uint32_t cluster_bar, int c0,
                                                 int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at `bar`'s offset in every CTA of `cta_mask`
// when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets row (lane base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 consecutive 32-bit TMEM columns of this thread's lane <-> 16 registers
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
// Shared-memory descriptor of an unswizzled tile of 16-byte rows stored
// back to back (8-row core matrices 128 bytes apart; the tile is one core
// matrix wide, so both strides are 128 bytes).
__device__ __forceinline__ uint64_t smem_desc_rows16(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128u >> 4) << 16;
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor: fp32 accumulator, dense, A/B format code (kind::f16:
// 1 = bf16; kind::f8f6f4: 0 = e4m3), operand majorness (1 = MN-major), N, M.
// Instruction descriptor of the block-scaled kind::mxf8f6f4 MMA: e4m3 A and B
// (format 0), both K-major, fp32 accumulator, M = m, N = n; bit 23 selects
// the scale format (1: ue8m0).  The scale-factor ids (bits 4-5 for B, 29-30
// for A: which byte of each 32-bit tensor-memory word the MMA takes) are
// or-ed in per MMA.
__host__ __device__ constexpr uint32_t make_idesc_mx(int m, int n, uint32_t ue8m0) {
  return ((uint32_t)(n >> 3) << 17) | ((ue8m0 & 1u) << 23) | ((uint32_t)(m >> 4) << 24);
}

__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, bool a_mn, bool b_mn, int m, int n) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// ---------------------------------------------------------------- numerics
// Power-of-two scale 2^floor(log2(fp32(448 / max(amax, 1e-12)))), with the
// floor taken from the exponent bits (exact).  The quotient is defined as the
// float64 quotient rounded once to fp32; a correctly rounded fp32 division
// gives the same fp32 value, because rounding first to 53 bits and then to 24
// cannot change a 24-bit quotient (53 >= 2 * 24 + 2).  The fp32 constant 1e-12f
// differs from the float64 one only in an interval that holds no bf16 value,
// and for amax below it the quotient (~4.48e14) sits far from a power-of-two
// boundary, so the power-of-two result is identical for every bf16 amax.
// (This GPU's float64 throughput is low; one fp32 division per value is cheap.)
__device__ __forceinline__ float pow2_scale_from_amax(float amax) {
  const float s = __fdiv_rn(448.0f, fmaxf(amax, 1e-12f));
  return __uint_as_float(__float_as_uint(s) & 0x7F800000u);
}

// Two floats -> two e4m3 bytes (round to nearest even, saturate to +-448).
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// ---------------------------------------------------------------- rows of bf16
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ float amax8(const uint4 &v, float a) {
  a = fmaxf(a, fabsf(bf16_lo(v.x)));
  a = fmaxf(a, fabsf(bf16_hi(v.x)));
  a = fmaxf(a, fabsf(bf16_lo(v.y)));
  a = fmaxf(a, fabsf(bf16_hi(v.y)));
  a = fmaxf(a, fabsf(bf16_lo(v.z)));
  a = fmaxf(a, fabsf(bf16_hi(v.z)));
  a = fmaxf(a, fabsf(bf16_lo(v.w)));
  a = fmaxf(a, fabsf(bf16_hi(v.w)));
  return a;
}

// 8 bf16 -> 8 e4m3 bytes (x * s is exact: s is a power of two)
__device__ __forceinline__ uint2 cast8(const uint4 &v, float s) {
  uint2 o;
  o.x = (uint32_t)cvt_e4m3x2(bf16_lo(v.x) * s, bf16_hi(v.x) * s) |
        ((uint32_t)cvt_e4m3x2(bf16_lo(v.y) * s, bf16_hi(v.y) * s) << 16);
  o.y = (uint32_t)cvt_e4m3x2(bf16_lo(v.z) * s, bf16_hi(v.z) * s) |
        ((uint32_t)cvt_e4m3x2(bf16_lo(v.w) * s, bf16_hi(v.w) * s) << 16);
  return o;
}

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// One row of C bf16 values (C % 8 == 0) -> e4m3 codes and its power-of-two
// scale, by one warp: the magnitude maximum in a first pass, the cast in a
// second (served by L2).  Loads go out eight chunks of 256 elements at a time.
__device__ __forceinline__ void quant_row_two_pass(const __nv_bfloat16 *src, int64_t C, uint8_t *dst, float *scale,
                                                   int lane) {
  float a = 0.f;
  for (int64_t c0 = 0; c0 < C; c0 += 8 * 256) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t c = c0 + i * 256 + lane * 8;
      v[i] = c < C ? ldg_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) a = amax8(v[i], a);
  }
  a = warp_max(a);
  const float s = pow2_scale_from_amax(a);
  if (lane == 0) *scale = s;
  for (int64_t c0 = 0; c0 < C; c0 += 8 * 256) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t c = c0 + i * 256 + lane * 8;
      v[i] = c < C ? *reinterpret_cast<const uint4 *>(src + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t c = c0 + i * 256 + lane * 8;
      if (c < C) *reinterpret_cast<uint2 *>(dst + c) = cast8(v[i], s);
    }
  }
}

// The same for a row of at most NCH * 256 elements held in registers between
// the two steps (one DRAM read).
template <int NCH>
__device__ __forceinline__ void quant_row_regs(const __nv_bfloat16 *src, int64_t C, uint8_t *dst, float *scale,
                                               int lane) {
  uint4 v[NCH];
  float a = 0.f;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int64_t c = ((int64_t)j * 32 + lane) * 8;
    v[j] = c < C ? ldg_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < NCH; ++j) a = amax8(v[j], a);
  a = warp_max(a);
  const float s = pow2_scale_from_amax(a);
  if (lane == 0) *scale = s;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int64_t c = ((int64_t)j * 32 + lane) * 8;
    if (c < C) *reinterpret_cast<uint2 *>(dst + c) = cast8(v[j], s);
  }
}

}  // namespace mgemm
