// mok_ptx.cuh -- inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA tile
// loads, and the tcgen05 tensor-core path (TMEM allocation, MMA issue, commit, TMEM loads).
//
// Every wait in this library is bounded: a wait that runs past its deadline records
// MOK_ERR_TIMEOUT in the device status word, raises the CTA's abort flag and returns false, so
// the kernel winds down and returns instead of hanging.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "mok.h"

namespace mok {

// ------------------------------------------------------------------------------------------------
// small helpers
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  Every kernel of the layer step starts with pdl_wait() and is
// launched with programmatic stream serialisation, so its CTAs may start launching as the previous
// kernel's last CTAs exit, before that grid's completion has been processed; pdl_wait() then holds
// them until the previous grid has completed and its memory is visible (it returns at once when
// there is no such dependency).  No kernel signals its dependents earlier than its exit: CTAs
// launched ahead of time to wait on an SM slowed the graph-replayed step.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Deadline of any single wait inside a kernel (ns).  Legitimate waits last microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void record_status(uint32_t* status, uint32_t code) {
  if (status) atomicOr(status, 1u << code);
}

// ------------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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
  return ok != 0;
}

// The same with cluster-scope acquire: for barriers that threads of the peer CTA arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (after recording a timeout and
// raising *abort) when the deadline passes or another role of the CTA has already aborted.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, uint32_t* status) {
  if (CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  while (true) {
    if (CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if ((++spins & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        record_status(status, MOK_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// clusters of two CTAs (a CTA pair sharing one tcgen05.mma.cta_group::2)
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of the variable at shared::cta address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}
// All threads of every CTA of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier given by its shared::cluster address (this CTA's or the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// ------------------------------------------------------------------------------------------------
// cluster launch control: a running CTA takes over the work of a CTA that has not started yet
// ------------------------------------------------------------------------------------------------
// Ask to cancel a not-yet-running CTA of this grid; the 16-byte answer lands at `resp` (16-byte
// aligned) and completes 16 bytes on mbarrier `bar`.  One thread; no new request after an answer
// that cancelled nothing.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
  asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];"
               ::"r"(resp), "r"(bar)
               : "memory");
}
// The x index of the CTA the answer at `resp` cancelled, or -1 when it cancelled none.
__device__ __forceinline__ int clc_cancelled_x(uint32_t resp) {
  uint32_t x, ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b128 r;\n\t"
      "mov.u32 %0, 0;\n\t"
      "ld.shared.b128 r, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %1, 1, 0, p;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, r;\n\t}"
      : "=r"(x), "=r"(ok)
      : "r"(resp)
      : "memory");
  return ok ? static_cast<int>(x) : -1;
}

// ------------------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) tile loads, completion counted on an mbarrier
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// c0 = innermost (contiguous) element coordinate, c1 = row coordinate.  c0 is always a multiple
// of 64 elements here, so the 16-byte rule on the inner coordinate holds.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Tile load into this CTA's shared memory whose completion is counted on an mbarrier of either CTA
// of the pair (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int32_t c0,
                                                 int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Tile store shared -> global (bulk-group completion).  Rows outside the tensor are clipped.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
// The same store marked evict-first in L2: for outputs nothing reads again soon (the forward
// context, weight gradients), so that they do not push out the operands other tiles reuse.
__device__ __forceinline__ void tma_store_2d_evict_first(const CUtensorMap* tm, uint32_t src, int32_t c0, int32_t c1) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;"
               ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(src), "r"(c0), "r"(c1), "l"(pol)
               : "memory");
}
// Untiled bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups still read their shared-memory sources.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk group has completed (global writes done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_u8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// ------------------------------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Pair forms: one warp of each CTA of the pair executes them together; the columns are allocated
// at the same address in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// CTA pair (issued by the first CTA of the pair only): M = 256 rows, A rows 0..127 from this CTA's
// shared memory and 128..255 from the peer's at the same address; B columns 0..N/2-1 from this
// CTA, N/2..N-1 from the peer; each CTA's TMEM receives the accumulator rows of its A rows.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= (A * SFA)[smem] * (B * SFB)[smem]^T with E4M3 A and B, one E8M0 scale per 32 K
// values (OCP MX), fp32 accumulation; K = 32 per instruction.  sfa_tmem / sfb_tmem address the TMEM
// columns holding the scale words of the A rows / B rows; the k-group byte used inside each 32-bit
// word is selected by the instruction descriptor (idesc_mx).
__device__ __forceinline__ void umma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate, uint32_t sfa_tmem, uint32_t sfb_tmem) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Copy one 512-byte scale atom (32 lines x 16 bytes) from shared memory to TMEM: line l lands in
// lane l of four consecutive columns, replicated into all four 32-lane quarters.  `sdesc` is a
// no-swizzle descriptor of the atom (sdesc_plain).
__device__ __forceinline__ void tmem_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Pair forms, issued by the first CTA of a CTA pair.  The copy moves each CTA's own shared-memory
// atom (same offset) into its own TMEM (same address).  The MMA is M = 256: each CTA's A rows and
// their scale words come from that CTA, B columns 0..N/2-1 from the first CTA and N/2..N-1 from the
// second, and each CTA's TMEM must hold the scale words of all N rows of B.
__device__ __forceinline__ void tmem_cp_sf_atom_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void umma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate, uint32_t sfa_tmem, uint32_t sfb_tmem) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Pair form: arrive once on the mbarrier at this shared-memory offset in both CTAs of the pair.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(bar), "h"(both)
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives TMEM lane
// (lane base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  descriptor version (1 on sm_100 family)
//   bits 49-51  base offset (0: every swizzle atom here starts 1024-byte aligned)
//   bit  52     leading-dimension offset mode (0: relative)
//   bits 61-63  swizzle mode (2: 128-byte swizzle)
// K-major operand (rows of 128 bytes = 64 bf16 along K): SBO = 1024 (8-row groups), LBO unused.
// MN-major operand (rows of 128 bytes = 64 bf16 along M or N, one row per k): LBO = distance
// between 64-element MN chunks, SBO = 1024 (8-k groups).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo_bytes & 0x3FFFFu) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Shared-memory descriptor without swizzle (16-byte lines; SBO = 128 between 8-line groups).
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale: E4M3 A and B (format 0), fp32
// D, UE8M0 scales (bit 23); bits 4-5 / 29-30 pick the byte (k-group) of the B / A scale words that
// this K = 32 step uses; bits 15 / 16: A / B MN-major (mn = both).
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t kgroup, bool mn = false) {
  return (kgroup << 4) | (mn ? (3u << 15) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24) | (kgroup << 29);
}

// Instruction descriptor of tcgen05.mma.kind::f16: bf16 A and B, fp32 D, dense.
//   bits 4-5 D format (1 = f32); 7-9 A format (1 = bf16); 10-12 B format (1 = bf16);
//   bit 15 A is MN-major; bit 16 B is MN-major; bits 17-22 N >> 3; bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------------------------------------
// MXFP8 helpers (OCP MX: E4M3 elements, one E8M0 scale per 32 values)
// ------------------------------------------------------------------------------------------------
// 2^e exactly, for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(1 << (e + 149));
}

// Larger magnitude of two fp32 values, NaN if either is NaN (one instruction); the sign of the
// result is the XOR of the operands' and means nothing here.
__device__ __forceinline__ float fmax_abs_nan(float a, float b) {
  float d;
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
// Bits of max |v[i]| over 32 values (a pairwise tree): above 0x7F7FFFFF means an Inf or a NaN.
__device__ __forceinline__ uint32_t absmax32_bits(const float* v) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmax_abs_nan(v[i], v[i + 16]);
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1) {
#pragma unroll
    for (int i = 0; i < s; ++i) m[i] = fmax_abs_nan(m[i], m[i + s]);
  }
  return __float_as_uint(m[0]) & 0x7FFFFFFFu;
}
// Two fp32 products in one instruction, each rounded as a single fp32 multiply.
__device__ __forceinline__ void fmul2(float& a, float& b, uint64_t s2) {
  asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%0, %1};\n\tmul.rn.f32x2 x, x, %2;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a), "+f"(b)
      : "l"(s2));
}
// (d0, d1) = (a0 * b0, a1 * b1) and (a0 * b0 + c0, a1 * b1 + c1) in one instruction each; every
// lane is rounded exactly as the scalar fp32 multiply or fused multiply-add.
__device__ __forceinline__ void mul_f32x2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmul.rn.f32x2 x, x, y;"
      "\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fma_f32x2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                          float c1) {
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\tmov.b64 z, {%6, %7};"
      "\n\tfma.rn.f32x2 x, x, y, z;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ uint64_t f32x2_splat(float s) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
  return r;
}

// MX quantisation of 32 fp32 values (one block): returns the E8M0 scale byte and writes the E4M3
// codes (byte i of the 32 = element i); with DEQ, v is replaced by the dequantised values.  shared
// = floor(log2 amax) - 8 (8 = the exponent of E4M3's largest normal), clamped below at -127 (amax 0
// or subnormal); codes = E4M3(v * 2^-shared), round to nearest even, saturating (the scaling by a
// power of two is exact in fp32).  A block holding a NaN or an infinity gets scale 0xFF and codes
// 0x7F (NaN), as the OCP MX format prescribes.
template <bool DEQ = true>
__device__ __forceinline__ uint32_t mx_quant32(float* v, uint32_t (&codes)[8]) {
  const uint32_t amax = absmax32_bits(v);
  if (amax > 0x7F7FFFFFu) {
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0x7F7F7F7Fu;
    if constexpr (DEQ) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __int_as_float(0x7FC00000);
    }
    return 0xFFu;
  }
  int shared = static_cast<int>(amax >> 23) - 127 - 8;
  shared = shared < -127 ? -127 : shared;
  const uint64_t dn2 = f32x2_splat(pow2f(-shared));
  const uint64_t up2 = f32x2_splat(pow2f(shared));
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float lo = v[2 * i], hi = v[2 * i + 1];
    fmul2(lo, hi, dn2);
    uint16_t q;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(hi), "f"(lo));
    if constexpr (DEQ) {
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q));
      lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
      hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
      fmul2(lo, hi, up2);
      v[2 * i] = lo;
      v[2 * i + 1] = hi;
    }
    if (i & 1) codes[i >> 1] |= static_cast<uint32_t>(q) << 16;
    else codes[i >> 1] = q;
  }
  return static_cast<uint32_t>(shared + 127);
}

// Byte offset of the scale of (row, k-group kg) in an atom-tiled MX scale array: 512-byte atoms of
// 128 rows x 4 k-groups, kq atoms per 128-row tile along K; inside an atom, row r's four bytes sit
// at (r % 32) * 16 + ((r / 32) % 4) * 4 -- the order in which tcgen05.cp's 32x128b.warpx4 shape
// puts them into TMEM for the block-scaled MMA.
__host__ __device__ __forceinline__ int64_t sf_atom_offset(int64_t row, int kg, int kq) {
  return ((row >> 7) * kq + (kg >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (kg & 3);
}

// Scale offset in an atom-tiled array whose rows are grouped G atoms at a time (G = 1 for an A
// operand, BN / 128 for a B operand read in BN-row tiles): row f (the operand's M or N index),
// k-group kg (K / 32), kq atoms per 128-row tile along K.  G = 1 equals sf_atom_offset.
__host__ __device__ __forceinline__ int64_t sf_atom_offset_g(int64_t f, int64_t kg, int64_t kq, int g) {
  return (((f / (128 * g)) * kq + (kg >> 2)) * g + (f >> 7) % g) * 512 + (f & 31) * 16 + ((f >> 5) & 3) * 4 +
         (kg & 3);
}

// sf_atom_offset_g for a power-of-two group count G = 1 << gl: shifts and masks instead of the
// 64-bit division and remainder (a called routine on the device).
__device__ __forceinline__ int64_t sf_atom_offset_p2(int64_t f, int64_t kg, int64_t kq, int gl) {
  const int64_t g = int64_t{1} << gl;
  return (((f >> (7 + gl)) * kq + (kg >> 2)) * g + ((f >> 7) & (g - 1))) * 512 + (f & 31) * 16 +
         ((f >> 5) & 3) * 4 + (kg & 3);
}

// bf16 helpers (round to nearest even, no special-value surprises for finite inputs)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

}  // namespace mok
