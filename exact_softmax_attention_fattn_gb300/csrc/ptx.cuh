// Thin inline-PTX wrappers for the sm_103a features the attention kernel uses:
// mbarriers, TMA tensor loads, tcgen05 (TMEM allocation, MMA, commit, ld/st)
// and the fences that order them.  Each wrapper is one PTX instruction (or a
// short fixed sequence); the semantics are those of the PTX ISA sections
// named beside them.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace fattn {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// True once the phase with the given parity has completed.
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

// Same, suspending the thread until the phase completes or about `hint_ns`
// nanoseconds have passed.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
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

// Non-suspending test of the same condition (no time-out hint, returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- TMA
// 3-D tiled tensor load into shared memory, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Tensor-memory allocation: executed by one full warp; writes the base address
// to shared memory.  ncols is a power of two >= 32.
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

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]  (kind::f16, one CTA)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]  (kind::f16, one CTA)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Warp-collective forms: the whole (converged) warp executes them with
// warp-uniform operands and elect.sync lets exactly one lane issue.
__device__ __forceinline__ void mma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same, with both descriptors advanced by the compile-time offset OFF (in
// 16-byte units) inside the instruction sequence.
template <uint32_t OFF>
__device__ __forceinline__ void mma_ss_w_off(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t.reg .b64 ad, bd;\n\t"
      "add.s64 ad, %1, %5;\n\t"
      "add.s64 bd, %2, %5;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(OFF)
      : "memory");
}

// Same, with the A and B descriptors advanced by different compile-time
// offsets (operand tiles whose panels differ in size).
template <uint32_t AOFF, uint32_t BOFF>
__device__ __forceinline__ void mma_ss_w_off2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t.reg .b64 ad, bd;\n\t"
      "add.s64 ad, %1, %5;\n\t"
      "add.s64 bd, %2, %6;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(AOFF), "n"(BOFF)
      : "memory");
}

// N SS MMAs over K = 16*N with one elect: both descriptors advanced along K
// (128-byte swizzled panels of 64 columns) in their low word only.
template <int N>
__device__ __forceinline__ void mma_ss_batch(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate);
template <>
__device__ __forceinline__ void mma_ss_batch<4>(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 alo, ahi, blo, bhi, al, bl;\n\t.reg .b64 ad, bd;\n\t"
      "mov.b64 {alo, ahi}, %1;\n\t"
      "mov.b64 {blo, bhi}, %2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.u32 al, alo, 2;\n\tadd.u32 bl, blo, 2;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 4;\n\tadd.u32 bl, blo, 4;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 6;\n\tadd.u32 bl, blo, 6;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
template <>
__device__ __forceinline__ void mma_ss_batch<8>(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 alo, ahi, blo, bhi, al, bl;\n\t.reg .b64 ad, bd;\n\t"
      "mov.b64 {alo, ahi}, %1;\n\t"
      "mov.b64 {blo, bhi}, %2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.u32 al, alo, 2;\n\tadd.u32 bl, blo, 2;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 4;\n\tadd.u32 bl, blo, 4;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 6;\n\tadd.u32 bl, blo, 6;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 1024;\n\tadd.u32 bl, blo, 1024;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 1026;\n\tadd.u32 bl, blo, 1026;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 1028;\n\tadd.u32 bl, blo, 1028;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 1030;\n\tadd.u32 bl, blo, 1030;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// O (+)= P V over 16*8 keys: P from tensor memory (16 keys = 8 columns), V MN-major.
__device__ __forceinline__ void mma_ts_batch8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 blo, bhi, bl, at;\n\t.reg .b64 bd;\n\t"
      "mov.b64 {blo, bhi}, %2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 bl, blo, 128;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 256;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 16;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 384;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 24;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 512;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 32;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 640;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 40;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 768;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 48;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 896;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 56;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same over 128 keys with A packed per 64-key half: keys 64h..64h+63 in
// TMEM columns 64h..64h+31 (two groups of threads, each packing its own half).
__device__ __forceinline__ void mma_ts_batch8_halves(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 blo, bhi, bl, at;\n\t.reg .b64 bd;\n\t"
      "mov.b64 {blo, bhi}, %2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 bl, blo, 128;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 256;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 16;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 384;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 24;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 512;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 64;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 640;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 72;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 768;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 80;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 896;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 88;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 SS MMAs over K = 256 behind one elect, A and B in 64-column panels of
// different sizes: A panels 16 KB apart (128-row tiles), B panels 8 KB apart
// (64-row tiles); descriptors advanced in their low word only.
__device__ __forceinline__ void mma_ss_batch16_a128_b64(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 alo, ahi, blo, bhi, al, bl;\n\t.reg .b64 ad, bd;\n\t"
      "mov.b64 {alo, ahi}, %1;\n\t"
      "mov.b64 {blo, bhi}, %2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.u32 al, alo, 2;\n\tadd.u32 bl, blo, 2;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 4;\n\tadd.u32 bl, blo, 4;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 6;\n\tadd.u32 bl, blo, 6;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 1024;\n\tadd.u32 bl, blo, 512;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 1026;\n\tadd.u32 bl, blo, 514;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 1028;\n\tadd.u32 bl, blo, 516;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 1030;\n\tadd.u32 bl, blo, 518;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 2048;\n\tadd.u32 bl, blo, 1024;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 2050;\n\tadd.u32 bl, blo, 1026;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 2052;\n\tadd.u32 bl, blo, 1028;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 2054;\n\tadd.u32 bl, blo, 1030;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 3072;\n\tadd.u32 bl, blo, 1536;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 3074;\n\tadd.u32 bl, blo, 1538;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 3076;\n\tadd.u32 bl, blo, 1540;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "add.u32 al, alo, 3078;\n\tadd.u32 bl, blo, 1542;\n\tmov.b64 ad, {al, ahi};\n\tmov.b64 bd, {bl, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, t;\n\t"
      "}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 4 TS MMAs over 64 keys behind one elect: A (P) from tensor memory, 16 keys
// = 8 columns; B (V, MN-major) 16 rows = 2048 bytes per step.
__device__ __forceinline__ void mma_ts_batch4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 blo, bhi, bl, at;\n\t.reg .b64 bd;\n\t"
      "mov.b64 {blo, bhi}, %2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %4, %4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 bl, blo, 128;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 8;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 256;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 16;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "add.u32 bl, blo, 384;\n\tmov.b64 bd, {bl, bhi};\n\tadd.u32 at, %1, 24;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, t;\n\t"
      "}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// TS form with the B descriptor advanced by OFF and the A TMEM column by ACOL.
template <uint32_t OFF, uint32_t ACOL>
__device__ __forceinline__ void mma_ts_w_off(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t.reg .b64 bd;\n\t.reg .b32 at;\n\t"
      "add.s64 bd, %2, %5;\n\t"
      "add.u32 at, %1, %6;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], bd, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(OFF), "n"(ACOL)
      : "memory");
}

__device__ __forceinline__ void mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Wait for this thread's outstanding tcgen05.ld; the registers are passed
// through so that no use of them can be scheduled above the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
        "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// 128 consecutive 32-bit TMEM columns of this warp's 32 lanes -> 128 registers per thread.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr));
}

// Wait for outstanding tcgen05.ld of 128 registers (tied so no use moves above the wait).
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63]), "+r"(r[64]), "+r"(r[65]), "+r"(r[66]), "+r"(r[67]), "+r"(r[68]), "+r"(r[69]), "+r"(r[70]), "+r"(r[71]), "+r"(r[72]), "+r"(r[73]), "+r"(r[74]), "+r"(r[75]), "+r"(r[76]), "+r"(r[77]), "+r"(r[78]), "+r"(r[79]), "+r"(r[80]), "+r"(r[81]), "+r"(r[82]), "+r"(r[83]), "+r"(r[84]), "+r"(r[85]), "+r"(r[86]), "+r"(r[87]), "+r"(r[88]), "+r"(r[89]), "+r"(r[90]), "+r"(r[91]), "+r"(r[92]), "+r"(r[93]), "+r"(r[94]), "+r"(r[95]), "+r"(r[96]), "+r"(r[97]), "+r"(r[98]), "+r"(r[99]), "+r"(r[100]), "+r"(r[101]), "+r"(r[102]), "+r"(r[103]), "+r"(r[104]), "+r"(r[105]), "+r"(r[106]), "+r"(r[107]), "+r"(r[108]), "+r"(r[109]), "+r"(r[110]), "+r"(r[111]), "+r"(r[112]), "+r"(r[113]), "+r"(r[114]), "+r"(r[115]), "+r"(r[116]), "+r"(r[117]), "+r"(r[118]), "+r"(r[119]), "+r"(r[120]), "+r"(r[121]), "+r"(r[122]), "+r"(r[123]), "+r"(r[124]), "+r"(r[125]), "+r"(r[126]), "+r"(r[127])
      :
      : "memory");
}

// 64 consecutive 32-bit TMEM columns of this warp's 32 lanes -> 64 registers per thread.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
      :
      : "memory");
}

// 64 consecutive fp32 TMEM columns -> 64 registers per thread, plus their
// maximum (the load's built-in max reduction, sm_103a).
__device__ __forceinline__ void tmem_ld64_max(uint32_t taddr, float (&r)[64], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x64.max.f32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, %64, [%65];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]), "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15]), "=f"(r[16]), "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]), "=f"(r[24]), "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]), "=f"(r[31]), "=f"(r[32]), "=f"(r[33]), "=f"(r[34]), "=f"(r[35]), "=f"(r[36]), "=f"(r[37]), "=f"(r[38]), "=f"(r[39]), "=f"(r[40]), "=f"(r[41]), "=f"(r[42]), "=f"(r[43]), "=f"(r[44]), "=f"(r[45]), "=f"(r[46]), "=f"(r[47]), "=f"(r[48]), "=f"(r[49]), "=f"(r[50]), "=f"(r[51]), "=f"(r[52]), "=f"(r[53]), "=f"(r[54]), "=f"(r[55]), "=f"(r[56]), "=f"(r[57]), "=f"(r[58]), "=f"(r[59]), "=f"(r[60]), "=f"(r[61]), "=f"(r[62]), "=f"(r[63]), "=f"(mx)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait(float (&r)[64], float& mx) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+f"(r[0]), "+f"(r[1]), "+f"(r[2]), "+f"(r[3]), "+f"(r[4]), "+f"(r[5]), "+f"(r[6]), "+f"(r[7]), "+f"(r[8]), "+f"(r[9]), "+f"(r[10]), "+f"(r[11]), "+f"(r[12]), "+f"(r[13]), "+f"(r[14]), "+f"(r[15]), "+f"(r[16]), "+f"(r[17]), "+f"(r[18]), "+f"(r[19]), "+f"(r[20]), "+f"(r[21]), "+f"(r[22]), "+f"(r[23]), "+f"(r[24]), "+f"(r[25]), "+f"(r[26]), "+f"(r[27]), "+f"(r[28]), "+f"(r[29]), "+f"(r[30]), "+f"(r[31]), "+f"(r[32]), "+f"(r[33]), "+f"(r[34]), "+f"(r[35]), "+f"(r[36]), "+f"(r[37]), "+f"(r[38]), "+f"(r[39]), "+f"(r[40]), "+f"(r[41]), "+f"(r[42]), "+f"(r[43]), "+f"(r[44]), "+f"(r[45]), "+f"(r[46]), "+f"(r[47]), "+f"(r[48]), "+f"(r[49]), "+f"(r[50]), "+f"(r[51]), "+f"(r[52]), "+f"(r[53]), "+f"(r[54]), "+f"(r[55]), "+f"(r[56]), "+f"(r[57]), "+f"(r[58]), "+f"(r[59]), "+f"(r[60]), "+f"(r[61]), "+f"(r[62]), "+f"(r[63]), "+f"(mx)
      :
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait_plain() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 registers per thread -> 32 consecutive 32-bit TMEM columns of this warp's lanes.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 16 registers per thread -> 16 consecutive 32-bit TMEM columns of this warp's lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- registers
// Per-warpgroup register reallocation; every warp of the warpgroup executes
// the same instruction.  N is a multiple of 8 in [24, 256].
template <int N>
__device__ __forceinline__ void regs_grow() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_shrink() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- dependent launch
// A kernel launched as a programmatic dependent of the previous one in its
// stream may start before that one ends: the previous kernel lets it launch
// (launch_dependents), and it waits (wait) for the previous kernel's
// completion and memory before reading what that kernel wrote.  Both are
// no-ops outside such a launch.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- math
// Packed pairs of fp32 (sm_100+ f32x2 arithmetic: one instruction, two lanes of work).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max of three (one instruction on sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Hardware base-2 exponential (MUFU), flush-to-zero; ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 bytes to global memory in one store (the address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                             uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0), "r"(a1), "r"(a2),
               "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// Two floats -> packed f16x2, round-to-nearest-even; `lo` lands in bits 0-15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> packed bf16x2, round-to-nearest-even; `lo` lands in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The two halves of a packed bf16x2 widened exactly to fp32 (a bf16 is the
// upper 16 bits of the fp32 with the same value).
__device__ __forceinline__ float bf16lo_as_f32(uint32_t b2) { return __uint_as_float(b2 << 16); }
__device__ __forceinline__ float bf16hi_as_f32(uint32_t b2) { return __uint_as_float(b2 & 0xFFFF0000u); }

// Packed f16x2 -> packed bf16x2 (each half widened exactly, then rounded to
// nearest even).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h2) {
  uint32_t r;
  asm("{\n\t.reg .f16 lo, hi;\n\t.reg .f32 flo, fhi;\n\t"
      "mov.b32 {lo, hi}, %1;\n\t"
      "cvt.f32.f16 flo, lo;\n\t"
      "cvt.f32.f16 fhi, hi;\n\t"
      "cvt.rn.bf16x2.f32 %0, fhi, flo;\n\t}"
      : "=r"(r)
      : "r"(h2));
  return r;
}

}  // namespace fattn
