// Shared device helpers for the qmoe kernels: inline PTX for mbarriers, bulk and
// tensor TMA copies, tcgen05 (TMEM allocation, MMA, loads, stores) and bounded
// waits.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmoe.h"

namespace qmoe {

// Error word layout at the start of every workspace.
struct ErrWord {
  unsigned int flags;
};

constexpr int kWsHeaderBytes = 256;
constexpr long long kWaitLimitNs = 2000000000LL;  // 2 s: no healthy wait comes close

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
// try_wait that lets the hardware suspend the thread for up to `hint_ns` while the
// phase is incomplete (the thread resumes as soon as it completes): waiting warps
// sleep instead of spinning through issue slots other warps need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's abort
// flag and the timeout bit of the error word) when `limit_ns` passes, or when
// another thread of the CTA has already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err, long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity, 200000u)) return true;
    if ((i & 3) == 0) {
      if (*abort_flag) return false;
      if ((long long)(globaltimer_ns() - t0) > limit_ns) {
        *abort_flag = 1;
        if (err) atomicOr(err, QMOE_FLAG_TIMEOUT);
        return false;
      }
    }
  }
}

// mbar_wait by every lane of a converged warp, with one warp-wide answer (so that a
// timeout seen by one lane cannot split the warp before an aligned instruction).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err));
}

// One lane of a converged warp; used as a predicate so that the single-thread
// instructions below (TMA, MMA, commit) are issued once while the warp's control
// flow stays uniform (issuing the copies from a divergent single thread was several
// times slower; the decode MMAs, whose operands the compiler can keep uniform, measured
// fewer instructions inside the elected lane's branch).
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred;
}

__device__ __forceinline__ void mbar_arrive_expect_tx_if(uint32_t pred, uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], %2;\n\t}" ::"r"(pred),
      "r"(bar), "r"(bytes)
      : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}


__device__ __forceinline__ void bulk_g2s_if(uint32_t pred, uint32_t dst, const void* src, uint32_t bytes,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%1], [%2], %3, [%4], %5;\n\t}" ::"r"(pred),
      "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_if(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                               int x, int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%1], [%2, {%3, %4}], [%5], %6;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 3-D tiled tensor copy by one lane (pred != 0); x (innermost) must be a multiple of
// 8 bf16 elements.
__device__ __forceinline__ void tma_load_3d_if(uint32_t pred, uint32_t dst, const CUtensorMap* map,
                                               int x, int y, int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%1], [%2, {%3, %4, %5}], [%6], %7;\n\t}" ::"r"(pred),
      "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}


__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- programmatic launch
// The forward's kernels after route are launched with programmatic stream
// serialization: a kernel may start while its predecessor finishes.  grid_dep_wait()
// blocks the calling thread until the predecessor grid has completed and its memory is
// visible (a no-op for a launch without the attribute); a thread must call it before
// it reads anything the predecessor writes.  grid_dep_launch() lets the successor be
// scheduled (as soon as every CTA of this grid has called it or exited).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
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
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this thread
// completes; issued only where pred != 0.
__device__ __forceinline__ void tc_commit_if(uint32_t pred, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}" ::"r"(
          pred),
      "r"(bar)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16 (bf16 inputs, fp32 accumulate), issued
// only where pred != 0 (one elected lane of a converged warp).
__device__ __forceinline__ void mma_bf16_ts_if(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem,
                                               uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %0, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %3, %4, q;\n\t}" ::"r"(pred),
      "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The 8 MMAs of one 128-wide K step in one block, issued by the elected lane:
// D (+)= A[a_tmem + 8j] * B[desc + 2j] for j = 0..7 (16-wide K slices; the B slices
// 2..3 and 4..7 sit in a second 64-wide slab `slab16` 16-byte units further on).
// Only the first MMA can start a fresh accumulation.  Keeping the issue to about
// three instructions per MMA matters: the issuing warp shares its scheduler with
// dequant warps, and the MMA pipe runs dry while it executes anything else.
__device__ __forceinline__ void mma_bf16_ts_step8(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem,
                                                  uint32_t desc_lo, uint32_t desc_hi,
                                                  uint32_t slab16, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q, t;\n\t.reg .b64 d;\n\t.reg .b32 lo, a;\n\t"
      "setp.ne.b32 p, %0, 0;\n\t"
      "setp.ne.b32 q, %7, 0;\n\t"
      "setp.eq.u32 t, 0, 0;\n\t"
      "mov.b64 d, {%3, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], d, %6, q;\n\t"
      "add.u32 lo, %3, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 8;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, %3, 4;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 16;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, %3, 6;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 24;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, %3, %5;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 32;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, lo, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 40;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, lo, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 48;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %6, t;\n\t"
      "add.u32 lo, lo, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 56;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %6, t;\n\t}" ::"r"(pred),
      "r"(d_tmem), "r"(a_tmem), "r"(desc_lo), "r"(desc_hi), "r"(slab16), "r"(idesc),
      "r"(accumulate)
      : "memory");
}

// The 4 MMAs of one 64-wide K slab: D (+)= A[a_tmem + 8j] * B[desc + 2j], j = 0..3.
// Only the first can start a fresh accumulation.
__device__ __forceinline__ void mma_bf16_ts_slab4(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem,
                                                  uint32_t desc_lo, uint32_t desc_hi,
                                                  uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q, t;\n\t.reg .b64 d;\n\t.reg .b32 lo, a;\n\t"
      "setp.ne.b32 p, %0, 0;\n\t"
      "setp.ne.b32 q, %6, 0;\n\t"
      "setp.eq.u32 t, 0, 0;\n\t"
      "mov.b64 d, {%3, %4};\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], d, %5, q;\n\t"
      "add.u32 lo, %3, 2;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 8;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %5, t;\n\t"
      "add.u32 lo, %3, 4;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 16;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %5, t;\n\t"
      "add.u32 lo, %3, 6;\n\tmov.b64 d, {lo, %4};\n\tadd.u32 a, %2, 24;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%1], [a], d, %5, t;\n\t}" ::"r"(pred),
      "r"(d_tmem), "r"(a_tmem), "r"(desc_lo), "r"(desc_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// As mma_bf16_ts_slab4 into two accumulators of one tile wider than 256 pairs: chain 0
// takes B rows 0..255 into d0, chain 1 the rows from 256 on (`off16` 16-byte units
// further on) into d1, alternating slice by slice so that each MMA of the narrow
// chain issues behind an independent one and its accumulation latency stays hidden.
__device__ __forceinline__ void mma_bf16_ts_slab4x2(uint32_t pred, uint32_t d0, uint32_t d1,
                                                    uint32_t a_tmem, uint32_t desc_lo,
                                                    uint32_t desc_hi, uint32_t off16,
                                                    uint32_t idesc0, uint32_t idesc1,
                                                    uint32_t accumulate) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = desc_lo + 2u * j;
    const uint64_t b0 = ((uint64_t)desc_hi << 32) | lo;
    const uint64_t b1 = ((uint64_t)desc_hi << 32) | (lo + off16);
    const uint32_t acc = j == 0 ? accumulate : 1u;
    mma_bf16_ts_if(pred, d0, a_tmem + 8u * j, b0, idesc0, acc);
    mma_bf16_ts_if(pred, d1, a_tmem + 8u * j, b1, idesc1, acc);
  }
}


__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// tcgen05.ld writes its registers asynchronously: they hold the data only after
// tcgen05.wait::ld.  The compiler sees the load's outputs as ready at once, so after
// the wait each loaded array goes through this empty statement, which it must treat as
// rewriting the registers: no use of them can then be scheduled above the wait.
__device__ __forceinline__ void tmem_ld_ready(uint32_t (&v)[16]) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15])
               :
               : "memory");
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                              // D format: f32
         | (1u << 7)                            // A format: bf16
         | (1u << 10)                           // B format: bf16
         | ((uint32_t)(N >> 3) << 17)           // N / 8
         | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte swizzled
// layout (rows of 128 bytes, 8-row groups 1024 bytes apart, groups 1024-aligned).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused here) = 16 B
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset = 1024 B
  d |= (uint64_t)1 << 46;                      // descriptor version
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}


}  // namespace qmoe
