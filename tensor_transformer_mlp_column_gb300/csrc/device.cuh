// device.cuh — inline-PTX building blocks for the sm_103a kernels:
// mbarriers with bounded waits, TMA tile loads, and the tcgen05 (5th-gen
// tensor core) allocation, MMA, commit and TMEM load instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace tpmlp {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tensor core).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrival without release semantics, for signals that order only
// tensor-memory reads already completed by tcgen05.wait::ld.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// The same test with a limit (ns) on how long the thread may be suspended
// inside the instruction while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait_for(uint32_t bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(suspend_ns)
      : "memory");
  return done != 0;
}
constexpr uint32_t kWaitSuspendNs = 20000;  // long waits sleep in the instruction instead of looping (0: its own limit)

// Shared state of one CTA's bounded waits.
struct WaitGuard {
  volatile int* abort_flag;  // shared memory: set once any wait of the CTA gives up
  uint64_t limit_ns;         // time limit of a single wait
  int* status;               // per-device status word in global memory
};

// Waits until the phase of `bar` with parity `parity` has completed. Gives up
// (returns false) when the wait exceeds the limit (then it raises the CTA's
// abort flag and records `site` in the status word) or when another thread of the
// CTA has already raised the abort flag.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, const WaitGuard& g, int site) {
  const uint32_t a = smem_addr(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (kWaitSuspendNs ? mbar_try_wait_for(a, parity, kWaitSuspendNs) : mbar_try_wait(a, parity)) return true;
    if ((it & 31u) == 0) {
      if (*g.abort_flag) return false;
      if (global_timer_ns() - t0 > g.limit_ns) {
        *g.abort_flag = 1;
        atomicCAS(g.status, 0, site);  // the first failure since the last check is the one reported
        return false;
      }
    }
  }
}

// Clean-up wait used after an abort: only the time limit ends it early.
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_addr(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ------------------------------------------------------------------ debug checks
//
// In the library's debug build (TPMLP_DEBUG defined), TPMLP_DCHECK(cond,
// status, check) tests an index or layout invariant on the device. A failed
// check records kSiteBoundsBase + check in the status word (if no earlier
// failure is recorded) and evaluates to false, and the caller skips the
// access the check guards, so the kernel neither traps nor touches memory out
// of range; tpmlp_check_status() then reports TPMLP_ERR_BOUNDS. In the normal
// build the macro is the constant true and the checks compile away.
#ifdef TPMLP_DEBUG
__device__ __forceinline__ bool debug_fail(int* status, int check) {
  if (status) atomicCAS(status, 0, kSiteBoundsBase + check);
  return false;
}
#define TPMLP_DCHECK(cond, status, check) ((cond) ? true : ::tpmlp::debug_fail((status), (check)))
#else
#define TPMLP_DCHECK(cond, status, check) true
#endif

// ------------------------------------------------------------------ dependent launch
//
// Kernels launched with programmatic stream serialisation may start while the
// previous kernel of the stream is still running: they set up shared memory,
// barriers and tensor memory, then wait here until that kernel has completed
// and its writes are visible, before touching global memory. Without the
// launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel of the stream start its own set-up.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk tensor load: box at (x = inner coordinate, y = outer
// coordinate) into shared memory, completing `bytes` on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// tma_load_2d with an L2 cache policy (l2_policy) for the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 3-D form of tma_load_2d_hint: box at (x, y, z).
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 2-D tiled bulk tensor store from this CTA's shared memory; the box at
// (x, y) is clipped to the tensor's bounds. Completion is tracked per thread
// with bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05

// Allocates `ncols` TMEM columns (power of two >= 32); whole warp. The TMEM
// address is written to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate; one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Loads 32 consecutive 32-bit TMEM columns of this warp's 32 lanes: thread t
// gets lane (base lane + t), columns col .. col+31.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Split form of tmem_ld_32cols for software pipelining: tmem_ld_32cols_issue
// starts the load, tmem_ld_wait waits for every load of the thread issued so
// far. The registers pass through the wait as operands, so no use of them can
// be scheduled before it.
__device__ __forceinline__ void tmem_ld_32cols_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// ------------------------------------------------------------------ CTA pairs (cta_group::2)

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
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Shared::cluster address of the object at the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Arrival on a barrier of another CTA of the cluster (cluster address), without release
// semantics: for signals that order only tensor-memory reads already
// completed by tcgen05.wait::ld, so the arrival need not wait for the
// thread's outstanding global stores.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// L2 eviction priority for a load, as a cache policy operand:
// 0 normal, 1 evict-last (keep: other CTAs read the same tile soon), 2 evict-first.
__device__ __forceinline__ uint64_t l2_policy(int kind) {
  uint64_t pol;
  if (kind == 1)
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  else if (kind == 2)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// TMA tile load into this CTA's shared memory whose completion is counted on
// a barrier that may live in the peer CTA (cluster address), with an L2 cache
// policy (l2_policy) for the loaded lines.
__device__ __forceinline__ void tma_load_2d_pair_hint(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                      uint32_t bar_cluster_addr, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr), "l"(policy)
      : "memory");
}

// 3-D form of tma_load_2d_pair_hint: box at (x, y, z).
__device__ __forceinline__ void tma_load_3d_pair_hint(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                      int32_t z, uint32_t bar_cluster_addr, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster_addr), "l"(policy)
      : "memory");
}

// TMEM allocation shared by the CTA pair: one warp of EACH CTA executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Pair MMA, issued by one thread of the even CTA: D (M=256 over both CTAs'
// TMEM) (+)= A (128 rows in each CTA) x B^T (N/2 rows in each CTA).
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the barrier at this offset in every CTA of `mask` when all
// pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// Shared-memory matrix descriptor for a K-major bf16 tile written by TMA with
// 128-byte swizzling: rows of 128 bytes (64 elements), 8-row swizzle atoms of
// 1024 bytes stacked along M/N (stride-dimension offset 1024 B). The leading
// offset is unused for this layout and set to 16 B. Bits 46..48 hold the
// fixed descriptor version 0b001; bits 61..63 the layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);        // start address
  d |= static_cast<uint64_t>(16u >> 4) << 16;                  // leading byte offset
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                        // version
  d |= static_cast<uint64_t>(2u) << 61;                        // 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor for an MN-major bf16 tile (M or N
// contiguous) with 128-byte swizzling, as TMA writes it from a row-major
// [K][MN] tensor in boxes of 64 MN elements x 64 K rows: each K row of a box
// is one 128-byte line (64 consecutive MN elements), 8 K rows form a
// 1024-byte swizzle atom. The stride-dimension offset steps from one group of
// 8 K rows to the next (1024 B); the leading offset steps from one 64-element
// MN chunk to the next, i.e. from one box to the next (8 KB apart). One
// K = 16 instruction reads 16 K rows, so successive instructions start
// 2048 bytes apart.
constexpr uint32_t kMnChunkBytes = 64 * 64 * 2;  // one 64 (MN) x 64 (K) box
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);        // start address
  d |= static_cast<uint64_t>(kMnChunkBytes >> 4) << 16;       // leading byte offset: next 64-element MN chunk
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                // stride byte offset: next 8 K rows
  d |= static_cast<uint64_t>(1u) << 46;                        // version
  d |= static_cast<uint64_t>(2u) << 61;                        // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32
// accumulator, shape M x N. a_mn / b_mn (bits 15 / 16) mark an operand held
// MN-major (M or N contiguous) instead of K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, uint32_t a_mn = 0, uint32_t b_mn = 0) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | ((a_mn & 1u) << 15)                       // A MN-major
         | ((b_mn & 1u) << 16)                       // B MN-major
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Descriptor of the K = 16 slice k (0..3) of one 64-deep K block of an
// operand tile at saddr: K-major tiles advance 32 bytes along the swizzled
// row, MN-major tiles 16 K rows (2048 bytes).
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr, int k, bool mn_major) {
  return mn_major ? smem_desc_sw128_mn(saddr + 2048u * static_cast<uint32_t>(k))
                  : smem_desc_sw128(saddr + 32u * static_cast<uint32_t>(k));
}

// ------------------------------------------------------------------ math

// GeLU of the GPT-2 tanh form, evaluated as x * sigmoid(2u), which equals
// 1/2 x (1 + tanh u) and keeps its relative accuracy for large negative x.
__device__ __forceinline__ float gelu_fast(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float k1 = 0.044715f;
  const float u = k0 * x * fmaf(k1, x * x, 1.0f);
  return __fdividef(x, 1.0f + __expf(-2.0f * u));
}

// GeLU for a result that is rounded to bf16: x/2 (1 + tanh u) with the
// hardware tanh approximation (tanh.approx.f32), one special-function
// instruction instead of the exponential and the reciprocal of gelu_fast,
// which halves the epilogue's special-function work. Its error, about
// 2^-11 |x| / 2 in absolute terms, is below bf16 rounding of the result except
// in the negative tail (x < -2), where the result itself is near zero.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float gelu_bf16_fast(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float k1 = 0.044715f;
  const float h = 0.5f * x;
  const float u = k0 * x * fmaf(k1, x * x, 1.0f);
  return fmaf(h, tanh_approx(u), h);
}

// GeLU and its derivative at x: with s = sigmoid(2u),
// GeLU = x s and GeLU' = s + 2 x s (1 - s) du/dx, du/dx = sqrt(2/pi)(1 + 3*0.044715 x^2).
__device__ __forceinline__ void gelu_and_grad_fast(float x, float& g, float& dg) {
  const float k0 = 0.7978845608028654f;
  const float k1 = 0.044715f;
  const float x2 = x * x;
  const float u = k0 * x * fmaf(k1, x2, 1.0f);
  const float s = __fdividef(1.0f, 1.0f + __expf(-2.0f * u));
  const float du = k0 * fmaf(3.0f * k1, x2, 1.0f);
  g = x * s;
  dg = fmaf(2.0f * x * s * (1.0f - s), du, s);
}

}  // namespace tpmlp
