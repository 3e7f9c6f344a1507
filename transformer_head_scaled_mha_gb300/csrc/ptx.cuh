// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tensor copies, tcgen05 tensor-memory (TMEM) allocation, MMA, loads and
// stores, and the shared-memory / instruction descriptors tcgen05.mma reads.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "common.cuh"

namespace mha {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// make barrier initialisation visible to the async proxy (TMA, tcgen05)
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Probe that may suspend the thread for up to `hint_ns` (it wakes as soon as
// the phase completes); returns whether the phase completed.
__device__ __forceinline__ bool mbar_try_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// non-blocking probe of a phase (test_wait never suspends the thread)
__device__ __forceinline__ bool mbar_probe(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete.  Gives up (returns
// false and sets the CTA's abort flag) after kWaitLimitNs of wall time, or at
// once when another warp of the CTA has given up.  The kernel reports an
// abort through the status word at its teardown.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// mbar_wait for a thread that must react at once: polls with test_wait,
// which never suspends the thread (try_wait may sleep for a while first).
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity,
                                               volatile int *abort_flag, uint64_t limit_ns) {
  if (mbar_probe(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_probe(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Warp-uniform bounded wait: every lane gets the same answer, so a warp
// never reaches a later collective instruction (tcgen05.ld/st, shuffles,
// barriers) with only part of its lanes.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity,
                                               volatile int *abort_flag, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, limit_ns));
}

// Teardown after a given-up wait: waits (at most 100 ms) for a phase that
// copies or products already in flight will complete, so the CTA's shared
// memory and TMEM outlive every access to them.
__device__ __forceinline__ bool wait_teardown(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity))
    if (global_timer_ns() - t0 > 100000000ull) return false;
  return true;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Blocks until the grid this launch depends on has completed and its memory
// operations are visible (a no-op when launched without the attribute).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next dependent launch in the stream start its CTAs early (they
// still run their own griddep_wait before touching global memory).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// fences
// ---------------------------------------------------------------------------
// generic-proxy shared-memory writes -> visible to the async proxy (TMA store,
// tcgen05.mma operand reads)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier over `nthreads` threads that also ANDs a predicate across
// them: every participant gets true only if all passed true.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tile mode
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Pulls the box at the given coordinates into L2 (no shared memory, no
// completion signal).
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap *map, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::
          "l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// all committed stores have finished reading shared memory
__device__ __forceinline__ void tma_store_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// all committed stores are complete
__device__ __forceinline__ void tma_store_wait0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory
// ---------------------------------------------------------------------------
// whole warp; writes the allocated TMEM base address to *dst (shared memory)
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
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

// Per-warpgroup register budget (all four warps of the warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16: A (M x 16 per step, bf16 pairs
// packed two per 32-bit column, row m in lane m) read from tensor memory
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// mbarrier arrives once all previously issued tcgen05 ops of this thread finish
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns: thread t of the warp gets lane
// (taddr.lane + t), columns taddr.col .. +31
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
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// 32 lanes x 32 bit, N = 1, 2, 4 or 8 consecutive columns
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[1]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r[0]) : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld16(taddr, r); }
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[1]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r[0])
               : "memory");
}
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[2]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1])
               : "memory");
}
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                   taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[16]) { tmem_st16(taddr, r); }

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor for tcgen05.mma.
//   [0,14)  start address >> 4
//   [16,30) leading-dimension byte offset >> 4
//   [32,46) stride-dimension byte offset >> 4
//   [46,48) descriptor version, 1 on sm_100-class parts
//   [49,52) base offset (0: every tile here starts 1024-byte aligned)
//   [61,64) layout: 2 = 128-byte swizzle
// Operand tiles here are rows of 128 bytes (64 bf16) written by TMA (or by
// threads) with the 128-byte swizzle; 8 rows form one 1024-byte atom.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// The two 32-bit halves of smem_desc_sw128: the low half holds the start
// address (>> 4) and the leading-dimension offset, the high half the stride
// offset, version and layout.  A later 16-byte-aligned piece of the same
// operand has the same high half and a low half larger by offset / 16 (no
// carry below 256 KiB of shared memory), so an issuing loop can keep the
// high half in one register and step the low half with one add.
__device__ __forceinline__ uint32_t smem_desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t smem_desc_hi(uint32_t sbo_bytes) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint64_t desc_join(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D.
//   [4,6) D format (1 = f32)  [7,10) A format (1 = bf16)  [10,13) B format
//   [15] A major (0 = K)  [16] B major (0 = K, 1 = MN)
//   [17,23) N >> 3  [24,29) M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}
// the same with A read MN-major as well (A stored with its M index contiguous)
__host__ __device__ constexpr uint32_t idesc_bf16_f32_amn(uint32_t M, uint32_t N, uint32_t b_mn_major) {
  return idesc_bf16_f32(M, N, b_mn_major) | (1u << 15);
}

// ---------------------------------------------------------------------------
// small numeric helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x for two bfloat16 values at once on the MUFU unit (one instruction for
// the pair); lo in the low half
__device__ __forceinline__ uint32_t ex2_bf16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Pairs of fp32 in one 64-bit register: sm_100-class parts execute add, sub
// and mul on both halves with one f32x2 instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// three-input maximum (one instruction on sm_100-class parts)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Row softmax numerator over 128 scores held as raw fp32 bits in r[4][32]:
//   x_c = s_c * scale_log2, and -inf outside lo <= c < hi (when `mask`)
// returns max_c x_c; r is overwritten with x.  Reductions use a tree (3-input
// max, 16 independent chains) so the dependency depth is ~8, not 128.
__device__ __forceinline__ float scale_mask_max128(uint32_t (&r)[4][32], float scale_log2,
                                                   bool mask, int lo, int hi) {
  const uint64_t sc = f2_pack(scale_log2, scale_log2);
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    float a, b;
    f2_unpack(f2_mul(f2_pack(__uint_as_float(r[c >> 5][c & 31]),
                             __uint_as_float(r[c >> 5][(c + 1) & 31])),
                     sc),
              a, b);
    if (mask) {
      a = static_cast<unsigned>(c - lo) < static_cast<unsigned>(hi - lo) ? a : -INFINITY;
      b = static_cast<unsigned>(c + 1 - lo) < static_cast<unsigned>(hi - lo) ? b : -INFINITY;
    }
    r[c >> 5][c & 31] = __float_as_uint(a);
    r[c >> 5][(c + 1) & 31] = __float_as_uint(b);
  }
#define MHA_X(c) __uint_as_float(r[(c) >> 5][(c) & 31])
  float m[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    m[k] = fmax3(MHA_X(k), MHA_X(k + 16), MHA_X(k + 32));
    m[k] = fmax3(m[k], MHA_X(k + 48), MHA_X(k + 64));
    m[k] = fmax3(m[k], MHA_X(k + 80), MHA_X(k + 96));
    m[k] = fmaxf(m[k], MHA_X(k + 112));
  }
#undef MHA_X
  const float a = fmax3(m[0], m[1], m[2]), b = fmax3(m[3], m[4], m[5]);
  const float c = fmax3(m[6], m[7], m[8]), d = fmax3(m[9], m[10], m[11]);
  const float e = fmax3(m[12], m[13], m[14]);
  return fmax3(fmax3(a, b, c), fmax3(d, e, m[15]), -INFINITY);
}

// Raw-score variant for a positive scale: s_c -> -inf outside lo <= c < hi
// (when `mask`), returns max_c s_c (the scaled max is scale_log2 times it).
__device__ __forceinline__ float mask_max128(uint32_t (&r)[4][32], bool mask, int lo, int hi) {
  if (mask) {
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (static_cast<unsigned>(c - lo) >= static_cast<unsigned>(hi - lo))
        r[c >> 5][c & 31] = __float_as_uint(-INFINITY);
  }
#define MHA_X(c) __uint_as_float(r[(c) >> 5][(c) & 31])
  float m[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    m[k] = fmax3(MHA_X(k), MHA_X(k + 16), MHA_X(k + 32));
    m[k] = fmax3(m[k], MHA_X(k + 48), MHA_X(k + 64));
    m[k] = fmax3(m[k], MHA_X(k + 80), MHA_X(k + 96));
    m[k] = fmaxf(m[k], MHA_X(k + 112));
  }
#undef MHA_X
  const float a = fmax3(m[0], m[1], m[2]), b = fmax3(m[3], m[4], m[5]);
  const float c = fmax3(m[6], m[7], m[8]), d = fmax3(m[9], m[10], m[11]);
  const float e = fmax3(m[12], m[13], m[14]);
  return fmax3(fmax3(a, b, c), fmax3(d, e, m[15]), -INFINITY);
}

// 2^x for a pair of floats on the FMA pipes instead of the MUFU unit.  Range
// reduction as in Cody and Waite (exact in base 2): x is clamped to >= -126,
// n = round(x) comes from adding 1.5 * 2^23 (the sum's last bit is the units
// place), f = x - n lies in [-1/2, 1/2], 2^f is a cubic with the smallest
// largest relative error on that interval (7.5e-5; coefficients fitted by
// fit_exp2_poly.py next to the sources), and n is added to the result's
// exponent field: the shifted sum keeps n's two's complement in its low bits,
// so (bits(sum) << 23) is n << 23 modulo 2^32.  For x >= -125 the relative
// error stays below 7.5e-5; below, results are under 2^-125.  x must not be
// -inf (a clamped -inf gives 2^-126, not 0) nor NaN.
constexpr float kExp2Shift = 12582912.0f;  // 1.5 * 2^23
constexpr float kExp2C0 = 9.999280572e-01f;
constexpr float kExp2C1 = 6.932609677e-01f;
constexpr float kExp2C2 = 2.426111251e-01f;
constexpr float kExp2C3 = 5.517166853e-02f;
__device__ __forceinline__ void exp2_poly2(float &a, float &b) {
  const uint64_t x = f2_pack(fmaxf(a, -126.f), fmaxf(b, -126.f));
  const uint64_t shift = f2_pack(kExp2Shift, kExp2Shift);
  const uint64_t t = f2_add(x, shift);
  const uint64_t f = f2_sub(x, f2_sub(t, shift));
  uint64_t q = f2_fma(f2_pack(kExp2C3, kExp2C3), f, f2_pack(kExp2C2, kExp2C2));
  q = f2_fma(q, f, f2_pack(kExp2C1, kExp2C1));
  q = f2_fma(q, f, f2_pack(kExp2C0, kExp2C0));
  float tl, th, ql, qh;
  f2_unpack(t, tl, th);
  f2_unpack(q, ql, qh);
  a = __uint_as_float(__float_as_uint(ql) + (__float_as_uint(tl) << 23));
  b = __uint_as_float(__float_as_uint(qh) + (__float_as_uint(th) << 23));
}

// p_c = exp2(s_c * scale_log2 - m) in place, one packed FMA per pair (0 when
// !live); returns sum_c p_c.  kPoly: pairs 1 and 3 of every five take the
// exponential on the FMA pipes (exp2_poly2), the rest on the MUFU unit, so
// both units share the work (no score may then be -inf: unmasked tiles only).
template <bool kPoly = false>
__device__ __forceinline__ float exp2_fma_sum128(uint32_t (&r)[4][32], float scale_log2, float m,
                                                 bool live) {
  const uint64_t sc = f2_pack(scale_log2, scale_log2);
  const uint64_t nm = f2_pack(-m, -m);
  uint64_t acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0ull;
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    float a, b;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c >> 5][c & 31]),
                             __uint_as_float(r[c >> 5][(c + 1) & 31])),
                     sc, nm),
              a, b);
    if (kPoly && ((c >> 1) % 5 == 1 || (c >> 1) % 5 == 3)) {
      exp2_poly2(a, b);
      a = live ? a : 0.f;
      b = live ? b : 0.f;
    } else {
      a = live ? ex2_approx(a) : 0.f;
      b = live ? ex2_approx(b) : 0.f;
    }
    r[c >> 5][c & 31] = __float_as_uint(a);
    r[c >> 5][(c + 1) & 31] = __float_as_uint(b);
    acc[(c >> 1) & 7] = f2_add(acc[(c >> 1) & 7], f2_pack(a, b));
  }
  acc[0] = f2_add(acc[0], acc[1]);
  acc[2] = f2_add(acc[2], acc[3]);
  acc[4] = f2_add(acc[4], acc[5]);
  acc[6] = f2_add(acc[6], acc[7]);
  acc[0] = f2_add(acc[0], acc[2]);
  acc[4] = f2_add(acc[4], acc[6]);
  acc[0] = f2_add(acc[0], acc[4]);
  float lo, hi;
  f2_unpack(acc[0], lo, hi);
  return lo + hi;
}

// p_c = exp2(x_c - m) in place (0 when !live); returns sum_c p_c (16 partial
// sums, packed adds)
__device__ __forceinline__ float exp2_sum128(uint32_t (&r)[4][32], float m, bool live) {
  const uint64_t mm = f2_pack(m, m);
  uint64_t acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0ull;
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    float a, b;
    f2_unpack(f2_sub(f2_pack(__uint_as_float(r[c >> 5][c & 31]),
                             __uint_as_float(r[c >> 5][(c + 1) & 31])),
                     mm),
              a, b);
    a = live ? ex2_approx(a) : 0.f;
    b = live ? ex2_approx(b) : 0.f;
    r[c >> 5][c & 31] = __float_as_uint(a);
    r[c >> 5][(c + 1) & 31] = __float_as_uint(b);
    acc[(c >> 1) & 7] = f2_add(acc[(c >> 1) & 7], f2_pack(a, b));
  }
  acc[0] = f2_add(acc[0], acc[1]);
  acc[2] = f2_add(acc[2], acc[3]);
  acc[4] = f2_add(acc[4], acc[5]);
  acc[6] = f2_add(acc[6], acc[7]);
  acc[0] = f2_add(acc[0], acc[2]);
  acc[4] = f2_add(acc[4], acc[6]);
  acc[0] = f2_add(acc[0], acc[4]);
  float lo, hi;
  f2_unpack(acc[0], lo, hi);
  return lo + hi;
}

// two floats -> packed bf16x2 (round to nearest even); lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// one float -> bf16 bits (round to nearest even)
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void st_shared_u16(uint32_t saddr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(saddr), "h"(v) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(saddr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_global_v4(void *ptr, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// 16 bytes global -> shared without registers (cp.async, L2 only); complete
// after cp_async_commit and cp_async_wait_all in the issuing thread
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *gptr) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte
// swizzled tile (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B)
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace mha
