// sm103_ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the attention kernel uses:
// mbarriers, TMA tensor copies, tcgen05 tensor-memory allocation, MMA, loads/stores and fences,
// plus the shared-memory matrix and instruction descriptors the MMA reads.
//
// Conventions (PTX ISA, tcgen05 chapter):
//  * A TMEM address is (lane << 16) | column.  Warp w of a CTA may touch lanes 32*(w%4) .. +31.
//  * Shared-memory operand tiles are written by TMA with the 128-byte swizzle: rows of 128 bytes,
//    the 16-byte chunks of row r XOR-permuted by (r % 8), 8-row atoms of 1024 bytes.  Every tile
//    base is 1024-byte aligned so the descriptor's base-offset field stays 0.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace exattn {

// ------------------------------------------------------------------------------------------
// generic helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One lane of the (converged) warp is elected; warp-collective.
__device__ __forceinline__ bool elect_one() {
  uint32_t is_elected;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(is_elected));
  return is_elected != 0;
}

// Register budget moves between warpgroups (all warps of a warpgroup execute the same one).
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done;
}

// Three phases probed at once (independent try_waits in one block, so their latencies overlap);
// nonzero when all three have completed.
__device__ __forceinline__ uint32_t mbar_try_wait3(uint32_t b0, uint32_t p0, uint32_t b1,
                                                   uint32_t p1, uint32_t b2, uint32_t p2) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred q0, q1, q2;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
      "and.pred q0, q0, q1;\n\tand.pred q0, q0, q2;\n\t"
      "selp.u32 %0, 1, 0, q0;\n\t}"
      : "=r"(done)
      : "r"(b0), "r"(p0), "r"(b1), "r"(p1), "r"(b2), "r"(p2)
      : "memory");
  return done;
}

// ------------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Same, with an L2 eviction-priority hint (a policy from createpolicy).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int32_t c0, int32_t c1, int32_t c2,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
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

// Warm L2 with a 3-D tile (no shared-memory destination, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int32_t c0, int32_t c1,
                                                   int32_t c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Tiled bulk store of a shared-memory box to global memory (rows past the tensor's extent are
// clipped), tracked by the issuing thread's bulk-async group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store of this thread has read its shared-memory source.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05: tensor memory
// ------------------------------------------------------------------------------------------
// Whole-warp collective: allocate `ncols` TMEM columns, writing the base address to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
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

// Arrive once on `bar` when every tcgen05 async op this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc), 16-bit operands.
__device__ __forceinline__ void mma_f16_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem desc), 16-bit operands.
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 8-bit (e4m3) operand forms.
__device__ __forceinline__ void mma_f8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f8_ts(uint32_t d, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ---- MMA chains: all MMAs of one product in one asm block.  Issued this way the tensor core
// runs the attention kernel's S / P V alternation at its full rate (64 cycles per 128x128x16
// bf16 MMA, measured); the same MMAs issued one asm statement at a time ran at 92-113 cycles.
// The first MMA accumulates into D when acc0 != 0, the others always accumulate.  KIND: 0 =
// kind::f16, 1 = kind::f8f6f4.  The per-MMA descriptors are a base plus immediate
// offsets (template arguments, in 16-byte units for shared-memory descriptors and in columns
// for tensor-memory A operands), formed inside the asm block, so only the bases occupy
// registers in the issuing thread.  Offsets of MMAs past N are ignored.

template <int N, int KIND, int O1, int O2, int O3, int O4, int O5, int O6, int O7>
__device__ __forceinline__ void mma_chain_ss_off(uint32_t d, uint32_t idesc, uint32_t acc0, uint64_t a,
                                                  uint64_t b) {
  static_assert(N == 2 || N == 4 || N == 8, "MMA chain length");
  if constexpr (N == 2 && KIND == 0) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b64 a1; .reg .b64 b1;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %3, %5;\n\tadd.s64 b1, %4, %5;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "l"(a), "l"(b), "n"(O1)
      : "memory");
  }
  if constexpr (N == 2 && KIND == 1) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b64 a1; .reg .b64 b1;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %3, %5;\n\tadd.s64 b1, %4, %5;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "l"(a), "l"(b), "n"(O1)
      : "memory");
  }
  if constexpr (N == 4 && KIND == 0) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b64 a1, a2, a3; .reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %3, %5;\n\tadd.s64 b1, %4, %5;\n\t"
      "add.s64 a2, %3, %6;\n\tadd.s64 b2, %4, %6;\n\t"
      "add.s64 a3, %3, %7;\n\tadd.s64 b3, %4, %7;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "l"(a), "l"(b), "n"(O1), "n"(O2), "n"(O3)
      : "memory");
  }
  if constexpr (N == 4 && KIND == 1) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b64 a1, a2, a3; .reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %3, %5;\n\tadd.s64 b1, %4, %5;\n\t"
      "add.s64 a2, %3, %6;\n\tadd.s64 b2, %4, %6;\n\t"
      "add.s64 a3, %3, %7;\n\tadd.s64 b3, %4, %7;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a2, b2, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a3, b3, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "l"(a), "l"(b), "n"(O1), "n"(O2), "n"(O3)
      : "memory");
  }
  if constexpr (N == 8 && KIND == 0) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b64 a1, a2, a3, a4, a5, a6, a7; .reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %3, %5;\n\tadd.s64 b1, %4, %5;\n\t"
      "add.s64 a2, %3, %6;\n\tadd.s64 b2, %4, %6;\n\t"
      "add.s64 a3, %3, %7;\n\tadd.s64 b3, %4, %7;\n\t"
      "add.s64 a4, %3, %8;\n\tadd.s64 b4, %4, %8;\n\t"
      "add.s64 a5, %3, %9;\n\tadd.s64 b5, %4, %9;\n\t"
      "add.s64 a6, %3, %10;\n\tadd.s64 b6, %4, %10;\n\t"
      "add.s64 a7, %3, %11;\n\tadd.s64 b7, %4, %11;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "l"(a), "l"(b), "n"(O1), "n"(O2), "n"(O3), "n"(O4), "n"(O5), "n"(O6), "n"(O7)
      : "memory");
  }
  if constexpr (N == 8 && KIND == 1) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b64 a1, a2, a3, a4, a5, a6, a7; .reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %3, %5;\n\tadd.s64 b1, %4, %5;\n\t"
      "add.s64 a2, %3, %6;\n\tadd.s64 b2, %4, %6;\n\t"
      "add.s64 a3, %3, %7;\n\tadd.s64 b3, %4, %7;\n\t"
      "add.s64 a4, %3, %8;\n\tadd.s64 b4, %4, %8;\n\t"
      "add.s64 a5, %3, %9;\n\tadd.s64 b5, %4, %9;\n\t"
      "add.s64 a6, %3, %10;\n\tadd.s64 b6, %4, %10;\n\t"
      "add.s64 a7, %3, %11;\n\tadd.s64 b7, %4, %11;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a2, b2, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a3, b3, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a4, b4, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a5, b5, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a6, b6, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a7, b7, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "l"(a), "l"(b), "n"(O1), "n"(O2), "n"(O3), "n"(O4), "n"(O5), "n"(O6), "n"(O7)
      : "memory");
  }
}

template <int N, int KIND, int BSTEP, int O1, int O2, int O3, int O4, int O5, int O6, int O7>
__device__ __forceinline__ void mma_chain_ts_off(uint32_t d, uint32_t idesc, uint32_t acc0, uint32_t a,
                                                  uint64_t b) {
  static_assert(N == 2 || N == 4 || N == 8, "MMA chain length");
  if constexpr (N == 2 && KIND == 0) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b32 a1; .reg .b64 b1;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.u32 a1, %3, %5;\n\tadd.s64 b1, %4, %6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "r"(a), "l"(b), "n"(O1), "n"(1 * BSTEP)
      : "memory");
  }
  if constexpr (N == 2 && KIND == 1) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b32 a1; .reg .b64 b1;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.u32 a1, %3, %5;\n\tadd.s64 b1, %4, %6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%3], %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a1], b1, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "r"(a), "l"(b), "n"(O1), "n"(1 * BSTEP)
      : "memory");
  }
  if constexpr (N == 4 && KIND == 0) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b32 a1, a2, a3; .reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.u32 a1, %3, %5;\n\tadd.s64 b1, %4, %8;\n\t"
      "add.u32 a2, %3, %6;\n\tadd.s64 b2, %4, %9;\n\t"
      "add.u32 a3, %3, %7;\n\tadd.s64 b3, %4, %10;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "r"(a), "l"(b), "n"(O1), "n"(O2), "n"(O3), "n"(1 * BSTEP), "n"(2 * BSTEP), "n"(3 * BSTEP)
      : "memory");
  }
  if constexpr (N == 4 && KIND == 1) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b32 a1, a2, a3; .reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.u32 a1, %3, %5;\n\tadd.s64 b1, %4, %8;\n\t"
      "add.u32 a2, %3, %6;\n\tadd.s64 b2, %4, %9;\n\t"
      "add.u32 a3, %3, %7;\n\tadd.s64 b3, %4, %10;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%3], %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a1], b1, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a2], b2, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a3], b3, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "r"(a), "l"(b), "n"(O1), "n"(O2), "n"(O3), "n"(1 * BSTEP), "n"(2 * BSTEP), "n"(3 * BSTEP)
      : "memory");
  }
  if constexpr (N == 8 && KIND == 0) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b32 a1, a2, a3, a4, a5, a6, a7; .reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.u32 a1, %3, %5;\n\tadd.s64 b1, %4, %12;\n\t"
      "add.u32 a2, %3, %6;\n\tadd.s64 b2, %4, %13;\n\t"
      "add.u32 a3, %3, %7;\n\tadd.s64 b3, %4, %14;\n\t"
      "add.u32 a4, %3, %8;\n\tadd.s64 b4, %4, %15;\n\t"
      "add.u32 a5, %3, %9;\n\tadd.s64 b5, %4, %16;\n\t"
      "add.u32 a6, %3, %10;\n\tadd.s64 b6, %4, %17;\n\t"
      "add.u32 a7, %3, %11;\n\tadd.s64 b7, %4, %18;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "r"(a), "l"(b), "n"(O1), "n"(O2), "n"(O3), "n"(O4), "n"(O5), "n"(O6), "n"(O7), "n"(1 * BSTEP), "n"(2 * BSTEP), "n"(3 * BSTEP), "n"(4 * BSTEP), "n"(5 * BSTEP), "n"(6 * BSTEP), "n"(7 * BSTEP)
      : "memory");
  }
  if constexpr (N == 8 && KIND == 1) {
    asm volatile(
      "{\n\t.reg .pred p, t; .reg .b32 a1, a2, a3, a4, a5, a6, a7; .reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      "setp.ne.b32 p, %2, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
      "add.u32 a1, %3, %5;\n\tadd.s64 b1, %4, %12;\n\t"
      "add.u32 a2, %3, %6;\n\tadd.s64 b2, %4, %13;\n\t"
      "add.u32 a3, %3, %7;\n\tadd.s64 b3, %4, %14;\n\t"
      "add.u32 a4, %3, %8;\n\tadd.s64 b4, %4, %15;\n\t"
      "add.u32 a5, %3, %9;\n\tadd.s64 b5, %4, %16;\n\t"
      "add.u32 a6, %3, %10;\n\tadd.s64 b6, %4, %17;\n\t"
      "add.u32 a7, %3, %11;\n\tadd.s64 b7, %4, %18;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%3], %4, %1, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a1], b1, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a2], b2, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a3], b3, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a4], b4, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a5], b5, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a6], b6, %1, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a7], b7, %1, t;\n\t"
      "}"
      :: "r"(d), "r"(idesc), "r"(acc0), "r"(a), "l"(b), "n"(O1), "n"(O2), "n"(O3), "n"(O4), "n"(O5), "n"(O6), "n"(O7), "n"(1 * BSTEP), "n"(2 * BSTEP), "n"(3 * BSTEP), "n"(4 * BSTEP), "n"(5 * BSTEP), "n"(6 * BSTEP), "n"(7 * BSTEP)
      : "memory");
  }
}

// ---- TMEM <-> registers, shape 32x32b: thread t of the warp owns lane (base + t), and each
// .xN moves N consecutive 32-bit columns.
#define EXATTN_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                     "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define EXATTN_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                     "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : EXATTN_R8(0), EXATTN_R8(8), EXATTN_R8(16), EXATTN_R8(24)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      EXATTN_W8(0), EXATTN_W8(8), EXATTN_W8(16), EXATTN_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      EXATTN_W8(0), EXATTN_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef EXATTN_R8
#undef EXATTN_W8

// ------------------------------------------------------------------------------------------
// descriptors
// ------------------------------------------------------------------------------------------
// Shared-memory matrix descriptor (tcgen05 form): start address, leading- and stride-dimension
// byte offsets (all >> 4), the fixed version bits 46..48 = 0b001, base offset 0, and the
// swizzle mode in bits 61..63 (2 = 128-byte swizzle, 4 = 64-byte swizzle).
//  K-major, 128B swizzle: rows of 128 B along K; SBO = 1024 (next 8-row group); LBO unused.
//  MN-major, 128B swizzle: rows of 128 B along M/N, one row per K index; SBO = 1024 (next
//  8 K-rows), LBO = byte distance to the next 128-byte-wide block along M/N.
__host__ __device__ constexpr uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes,
                                                 uint32_t sbo_bytes, uint32_t swizzle_mode) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) |
         (static_cast<uint64_t>(1u) << 46) | (static_cast<uint64_t>(swizzle_mode & 7u) << 61);
}

constexpr uint32_t kSwizzle128B = 2;
constexpr uint32_t kSwizzle64B = 4;

// Instruction descriptor for kind::f16 and kind::f8f6f4 with fp32 accumulation:
// bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format, 15/16 A/B major (1 = MN-major),
// 17-22 N >> 3, 24-28 M >> 4.  A/B format: kind::f16 0 = f16, 1 = bf16; kind::f8f6f4 0 = e4m3.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t M, uint32_t N, uint32_t ab_format,
                                                  bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ------------------------------------------------------------------------------------------
// conversions and fast math
// ------------------------------------------------------------------------------------------
// Pack two fp32 into bf16x2 (round to nearest even): `lo` in bits 0-15, `hi` in bits 16-31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Pack two fp32 into f16x2 (round to nearest even): `lo` in bits 0-15, `hi` in bits 16-31.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^x for both halves of an f16x2 (MUFU, two results per instruction).
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Sum of two f16x2, element by element (round to nearest even).
__device__ __forceinline__ uint32_t hadd_f16x2(uint32_t a, uint32_t b) {
  uint32_t y;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
  return y;
}

// The two halves of an f16x2 as fp32 (exact): bits 0-15 -> .x, bits 16-31 -> .y.
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
  float lo, hi;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  return make_float2(lo, hi);
}

// Four f16 values (a: bits 0-15 -> byte 0, bits 16-31 -> byte 1; b likewise -> bytes 2-3) times
// 2^8 (exact in f16), rounded to e4m3 (nearest even, saturating).
__device__ __forceinline__ uint32_t e4m3x4_from_f16x2_scaled256(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("{\n\t.reg .b32 sa, sb, k;\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 k, 0x5C005C00;\n\t"
      "mul.rn.f16x2 sa, %1, k;\n\t"
      "mul.rn.f16x2 sb, %2, k;\n\t"
      "cvt.rn.satfinite.e4m3x2.f16x2 lo, sa;\n\t"
      "cvt.rn.satfinite.e4m3x2.f16x2 hi, sb;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "r"(a), "r"(b));
  return r;
}

// Widen two e4m3 values (byte 0 -> bits 0-15, byte 1 -> bits 16-31) to f16x2; exact, since
// every e4m3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Pack four fp32 into e4m3x4 (round to nearest even, saturating): a in byte 0 .. d in byte 3.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// Packed fp32 pairs: Blackwell executes fma/add/mul on both halves of a register pair in one
// instruction, each half rounded exactly as the scalar operation.  The compiler's float2
// builtins are used (not inline asm), so it can place the pairs in registers itself.
__device__ __forceinline__ float2 f32x2(float lo, float hi) { return make_float2(lo, hi); }
__device__ __forceinline__ float f32x2_lo(float2 v) { return v.x; }
__device__ __forceinline__ float f32x2_hi(float2 v) { return v.y; }
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
  return __ffma2_rn(a, b, c);
}
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// max of three floats in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Hardware 2^x (MUFU), flush-to-zero; 2^-inf = +0.
__device__ __forceinline__ float ex2_mufu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x on the FMA pipe ("FlashAttention4 精读", section 3.1.3): x = n + f with n = floor(x) taken
// by adding the magic bias 1.5 * 2^23 with round-down, 2^f from a degree-3 polynomial with
// constant term 1 in Horner form, and n added to the exponent field of the result.  Inputs are
// clamped to >= -126 so 2^n stays normal (a masked -inf input gives 2^-126, not 0; callers that
// mask must select 0 themselves).  Coefficients: minimax fit of the relative error on [0, 1)
// (fit_exp2_poly.py), max relative error 8.6e-5 in fp32.
__device__ __forceinline__ float ex2_poly(float x) {
  constexpr float kA1 = 0.6951167583465576f;
  constexpr float kA2 = 0.22764499485492706f;
  constexpr float kA3 = 0.07706703990697861f;
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  x = fmaxf(x, -126.0f);
  const float t = __fadd_rd(x, kMagic);
  const float f = x - (t - kMagic);
  float p = fmaf(kA3, f, kA2);
  p = fmaf(p, f, kA1);
  p = fmaf(p, f, 1.0f);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

__device__ __forceinline__ float lg2_mufu(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace exattn
