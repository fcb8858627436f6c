// ptx.cuh — hand-written inline-PTX building blocks for sm_103a.
//
// mbarrier, TMA (cp.async.bulk.tensor) and 5th-generation tensor-core
// (tcgen05) wrappers used by the attention kernel.  Every wait a kernel does
// on an mbarrier goes through wait_bounded(), which gives up after a time
// bound (read from %globaltimer) or when another role of the same CTA has
// already given up, so that no wait can spin forever.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda.h>  // CUtensorMap

namespace ea {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
// All shared-memory operands are 32-bit shared-window addresses (smem_u32);
// pointer overloads are provided for convenience.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended for up to `hint_ns` while
// the phase is incomplete (it resumes as soon as the phase completes), so a
// waiting warp does not take issue slots from the warps that compute.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ int ld_volatile_shared(uint32_t addr) {
  int v;
  asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_volatile_shared(uint32_t addr, int v) {
  asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// What a bounded wait needs: the CTA's abort flag (shared memory, non-zero
// once any role gave up), the global status words, and the bound.
struct WaitCtl {
  uint32_t abort_flag;  // shared-window address of an int
  int* status;          // global status words [error bits, first wait site] (may be null)
  uint64_t timeout_ns;  // bound on one wait
};

// Longest a bounded wait lets a thread sleep inside one try_wait (it wakes as
// soon as the phase completes); the timeout and abort flag are checked between.
constexpr uint32_t kSuspendHintNs = 200000;

// Device status bits (combined with atomicOr in the global status word).
enum : int { kStatusTimeout = 1, kStatusBounds = 2 };

static __device__ __noinline__ void raise_abort(const WaitCtl& c, int where) {
  st_volatile_shared(c.abort_flag, 1);
  if (c.status != nullptr) {
    atomicOr(c.status, kStatusTimeout);
    atomicCAS(c.status + 1, 0, where);  // first place that gave up, for diagnosis
  }
}

// Wait for the phase of `bar` with parity `parity` to complete.  Returns false
// if it did not complete within c.timeout_ns or if the CTA is aborting; in
// the first case the abort is raised here.  `where` tags the wait site.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                             int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_suspend(bar, parity, kSuspendHintNs)) return true;
    if (ld_volatile_shared(c.abort_flag)) return false;
    if (global_timer_ns() - t0 > c.timeout_ns) {
      raise_abort(c, where);
      return false;
    }
  }
}

// ---------------------------------------------------------------- debug checks
// Built with -DATTN_DEBUG, the kernels check the index arithmetic of each
// memory access before making it: TMA coordinates (16-byte column alignment,
// boxes that start inside the tensor), shared- and tensor-memory addresses
// against the CTA's allocation, and the row and column of every plain global
// load or store.  A failed check sets kStatusBounds and the site in the
// status words, and the access is skipped, so a bad index never reaches
// memory.  Release builds compile every check to `true`.
#ifdef ATTN_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

struct DbgBounds {
  int* status;        // status words (may be null)
  uint32_t smem_lo;   // the CTA's dynamic shared memory, [smem_lo, smem_hi)
  uint32_t smem_hi;
  int rows;           // rows of one (b, h) slice: S
  int cols;           // columns of the 16-bit tensors: the head dimension
  int slices;         // B·H
};

static __device__ __noinline__ void dbg_fail(int* status, int site) {
  if (status != nullptr) {
    atomicOr(status, kStatusBounds);
    atomicCAS(status + 1, 0, site);
  }
}

__device__ __forceinline__ bool dbg(bool ok, const DbgBounds& d, int site) {
  if (!kDebugChecks || ok) return true;
  dbg_fail(d.status, site);
  return false;
}

// `bytes` of shared memory at `addr`, aligned to `align` (a power of two).
__device__ __forceinline__ bool dbg_smem(const DbgBounds& d, uint32_t addr, uint32_t bytes,
                                         uint32_t align, int site) {
  if (!kDebugChecks) return true;
  return dbg(addr >= d.smem_lo && addr + bytes <= d.smem_hi && (addr & (align - 1)) == 0, d, site);
}

// A tiled TMA copy of a 128-byte-swizzled box into (or out of) `bytes` of
// shared memory at `saddr`, at tensor coordinates (x, y, z): x a multiple of 8
// 16-bit values (16 bytes) and not negative, the box's first row and slice
// inside the tensor (a load may run past the end and reads zeros there; a
// store must start inside the tensor's columns too).
__device__ __forceinline__ bool dbg_tma(const DbgBounds& d, uint32_t saddr, uint32_t bytes, int x,
                                        int y, int z, bool store, int site) {
  if (!kDebugChecks) return true;
  const bool coords = x >= 0 && (x & 7) == 0 && y >= 0 && y < d.rows && z >= 0 && z < d.slices &&
                      (!store || x < d.cols);
  return dbg(coords && saddr >= d.smem_lo && saddr + bytes <= d.smem_hi && (saddr & 1023) == 0, d,
             site);
}

// `ncols` tensor-memory columns from the address `taddr` (lane << 16 | column)
// of a 512-column allocation, in the lane quarter of warp `warp`.
__device__ __forceinline__ bool dbg_tmem(const DbgBounds& d, uint32_t taddr, uint32_t ncols,
                                         int warp, int site) {
  if (!kDebugChecks) return true;
  const uint32_t col = taddr & 0xffffu, lane = taddr >> 16;
  return dbg(col + ncols <= 512u && lane == 32u * static_cast<uint32_t>(warp & 3), d, site);
}

// The same for an MMA operand or accumulator (any lane quarter).
__device__ __forceinline__ bool dbg_tmem_cols(const DbgBounds& d, uint32_t taddr, uint32_t ncols,
                                              int site) {
  if (!kDebugChecks) return true;
  return dbg((taddr & 0xffffu) + ncols <= 512u && (taddr >> 16) == 0u, d, site);
}

// A check whose outcome a whole warp acts on (it guards a warp-collective
// instruction): every lane gets the warp's verdict.  Call with the full warp.
__device__ __forceinline__ bool dbg_warp(bool ok) {
  if (!kDebugChecks) return true;
  return __all_sync(0xffffffffu, ok);
}

// A plain global access of `n` 16-bit values at column `col` of row `row` of
// slice `bh`, or (n = 0) of one per-row fp32 value.
__device__ __forceinline__ bool dbg_row(const DbgBounds& d, int bh, int row, int col, int n,
                                        int site) {
  if (!kDebugChecks) return true;
  return dbg(bh >= 0 && bh < d.slices && row >= 0 && row < d.rows && col >= 0 && col + n <= d.cols,
             d, site);
}

// Wait used only while tearing down after an abort: ignores the abort flag,
// bounded by its own limit.  Returns false if the limit ran out.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// pointer overloads
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) { mbar_init(smem_u32(bar), count); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) { mbar_arrive(smem_u32(bar)); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  mbar_arrive_expect_tx(smem_u32(bar), bytes);
}
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, const WaitCtl& c,
                                             int where) {
  return wait_bounded(smem_u32(bar), parity, c, where);
}
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  return wait_drain(smem_u32(bar), parity, limit_ns);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load global → shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                            int y, int z, uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z),
        "l"(cache_policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, int z, uint64_t cache_policy) {
  tma_load_3d(smem_u32(dst), map, smem_u32(bar), x, y, z, cache_policy);
}

// 3-D tiled store shared → global (rows outside the tensor are not written).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                             int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}

// 16-byte read-only global load with an L2 cache policy (createpolicy).
__device__ __forceinline__ uint4 ldg_policy(const void* ptr, uint64_t policy) {
  uint4 r;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr), "l"(policy));
  return r;
}

// 3-D tiled store shared → global with an L2 cache policy.
__device__ __forceinline__ void tma_store_3d_policy(const CUtensorMap* map, uint32_t src, int x,
                                                    int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint"
      " [%0, {%2, %3, %4}], [%1], %5;"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

// Brings one box of a tiled tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Waits until every committed bulk store of this thread has finished reading
// its shared-memory source (the global writes may still be in flight).
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ---------------------------------------------------------------- cluster launch control
// A running CTA asks for the work of a CTA of the same grid that has not been
// launched yet: if granted, that CTA will never be launched and its index is
// handed over in a 16-byte response written to shared memory at `resp`
// (16-byte aligned), completing 16 transaction bytes on `bar` (which the
// caller arms with mbar_arrive_expect_tx(bar, 16) first).  Once a request has
// been refused, no further request may be made.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
      "[%0], [%1];" ::"r"(resp), "r"(bar)
      : "memory");
}

// Decodes a completed response: true and the granted CTA's x index, or false
// if the request was refused (no CTA left to hand over).
__device__ __forceinline__ bool clc_granted(uint32_t resp, int* first_x) {
  uint32_t ok, x;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
      "ld.shared.b128 r, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
      : "=r"(ok), "=r"(x)
      : "r"(resp)
      : "memory");
  *first_x = static_cast<int>(x);
  return ok != 0;
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tensor core) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- tcgen05
// Tensor-memory allocation (whole warp).  The TMEM address is written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  tmem_alloc(smem_u32(dst_smem), ncols);
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] · B[smem desc]; kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] · B[smem desc]; kind::f16.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// As mma_ts, mma_ss and mma_commit, executed by the whole (converged) warp: only the
// lane whose `issue` is true issues, so the warp never branches around them.
__device__ __forceinline__ void mma_ts_p(bool issue, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 e, %5, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue ? 1u : 0u)
      : "memory");
}
__device__ __forceinline__ void mma_ss_p(bool issue, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 e, %5, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue ? 1u : 0u)
      : "memory");
}
__device__ __forceinline__ void mma_commit_p(bool issue, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "setp.ne.b32 e, %1, 0;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
      ::"r"(bar), "r"(issue ? 1u : 0u) : "memory");
}

// TMEM[lanes 0-127, 8 columns from taddr] = a 128-row x 32-byte block of
// shared memory described by a matrix descriptor (the layout an MMA operand
// descriptor gives): row r lands in lane r, its 16 16-bit values two per
// column, which is the A-operand layout of a TS product.  Asynchronous, and
// executed in order with the tcgen05.mma this thread issues after it.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t s_desc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(s_desc) : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) { mma_commit(smem_u32(bar)); }

// 32 lanes x 32 bits, 32 consecutive columns: thread t of the warp gets
// lane (lane field of taddr + t), columns col .. col+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
        "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15])
      : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_st_words(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32) tmem_st_32x32b_x32(taddr, r);
  else tmem_st_32x32b_x16(taddr, r);
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// After tmem_ld_wait(): re-defines the registers so that no use of them can
// be scheduled before the wait.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

// One lane of the (fully active) warp is elected; the same lane every time.
__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(r));
  return r != 0;
}

// ---------------------------------------------------------------- registers
// Per-warpgroup register budget (all four warps of the warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void warpgroup_reg_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void warpgroup_reg_acquire() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two fp32 into bf16x2 (round to nearest even): lo → bits 0-15, hi → 16-31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Pack two fp32 into f16x2 (round to nearest even): lo → bits 0-15, hi → 16-31.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The 16-bit input type of the tensor-core operands: fp16 (F16) or bf16.
template <bool F16>
__device__ __forceinline__ uint32_t pack_x2(float lo, float hi) {
  if constexpr (F16) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

// x rounded to the 16-bit type (nearest even) and back to fp32.
template <bool F16>
__device__ __forceinline__ float round_to_x(float x) {
  const uint32_t v = pack_x2<F16>(x, 0.f) & 0xffffu;
  if constexpr (F16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v)));
  } else {
    return __uint_as_float(v << 16);
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d) : "memory");
}

}  // namespace ea
