// Inline-PTX wrappers for the fifth-generation tensor cores (tcgen05) on
// sm_103a: tensor-memory allocation, MMA issue with the accumulator in tensor
// memory, completion through mbarriers, tensor-memory loads and stores, and
// the shared-memory matrix and instruction descriptors of kind::f16 MMAs.
#pragma once

#include <stdint.h>

#include "rbkv_ptx.cuh"

namespace rbkv {
namespace tc {

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   ptx::smem_u32(slot)),
               "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   ptx::smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1, 128-byte swizzle.
// The kernels issue MMAs with its two 32-bit words (below); this 64-bit form
// is the definition the words are checked against.
__host__ __device__ constexpr uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);  // 128-byte swizzle
}

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}


// A descriptor split in its two 32-bit words.  Between operands of one
// layout only the start address (bits 0-13 of the low word, address >> 4)
// changes, so the issuing thread keeps one low word per operand base and adds
// (byte offset >> 4) for each MMA: one integer add instead of rebuilding the
// 64-bit descriptor.  Shared-memory addresses stay below 2^18, so the sum
// never carries out of the address field.
__host__ __device__ constexpr uint32_t desc_lo(uint32_t addr, uint32_t lbo) {
  return ((addr & 0x3FFFF) >> 4) | (((lbo >> 4) & 0x3FFF) << 16);
}
__host__ __device__ constexpr uint32_t desc_hi(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFF) | (1u << 14) | (2u << 29);   // version 1, 128-byte swizzle
}
static_assert((((uint64_t)desc_hi(1024) << 32) | desc_lo(0x2F3C0, 16)) ==
                  smem_desc(0x2F3C0, 16, 1024) &&
              (((uint64_t)desc_hi(1024) << 32) | desc_lo(0x08000, 16384)) ==
                  smem_desc(0x08000, 16384, 1024) &&
              desc_lo(0x08000, 16384) + (0x2000 >> 4) == desc_lo(0x0A000, 16384),
              "descriptor words must match the 64-bit descriptor");

// D[tmem] (+)= A[smem] * B[smem] with the descriptors given as words,
// kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void tc_mma_ss_w(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                            uint32_t hi, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.u32 p, %5, 0;\n\t"
      "mov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem] with B's descriptor given as words.  A is M
// rows = TMEM lanes, its K elements packed two per 32-bit column.
__device__ __forceinline__ void tc_mma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                            uint32_t hi, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "setp.ne.u32 p, %5, 0;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Eight MMAs over K = 128 (eight K = 16 steps) in one block, with the
// per-step operand offsets as immediates, so that nothing the compiler
// schedules sits between them.
// SS, both operands K-major with 128-byte swizzle and two 64-column halves
// 16 KB apart: step kk reads columns 16kk.. at byte offset (kk/4) * 16384 +
// (kk%4) * 32, i.e. descriptor address units 0, 2, 4, 6, 1024, ..., 1030.
__device__ __forceinline__ void tc_mma_ss_k128(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                               uint32_t hi, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b32 a, b;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.u32 p0, %5, 0;\n\tsetp.eq.u32 p1, %5, %5;\n\t"
      "mov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p0;\n\t"
      "add.u32 a, %1, 2;\n\tadd.u32 b, %2, 2;\n\tmov.b64 da, {a, %3};\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 a, %1, 4;\n\tadd.u32 b, %2, 4;\n\tmov.b64 da, {a, %3};\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 a, %1, 6;\n\tadd.u32 b, %2, 6;\n\tmov.b64 da, {a, %3};\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 a, %1, 1024;\n\tadd.u32 b, %2, 1024;\n\tmov.b64 da, {a, %3};\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 a, %1, 1026;\n\tadd.u32 b, %2, 1026;\n\tmov.b64 da, {a, %3};\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 a, %1, 1028;\n\tadd.u32 b, %2, 1028;\n\tmov.b64 da, {a, %3};\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t"
      "add.u32 a, %1, 1030;\n\tadd.u32 b, %2, 1030;\n\tmov.b64 da, {a, %3};\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p1;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// TS over K = 128: A (P, bf16 pairs) in tensor memory, step kk at column
// a_tmem + 8kk; B (V) MN-major with 128-byte swizzle, step kk 16 rows on,
// i.e. 2048 bytes = 128 descriptor address units.
__device__ __forceinline__ void tc_mma_ts_k128(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                               uint32_t hi, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b32 a, b;\n\t.reg .b64 db;\n\t"
      "setp.ne.u32 p0, %5, 0;\n\tsetp.eq.u32 p1, %5, %5;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p0;\n\t"
      "add.u32 a, %1, 8;\n\tadd.u32 b, %2, 128;\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %4, p1;\n\t"
      "add.u32 a, %1, 16;\n\tadd.u32 b, %2, 256;\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %4, p1;\n\t"
      "add.u32 a, %1, 24;\n\tadd.u32 b, %2, 384;\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %4, p1;\n\t"
      "add.u32 a, %1, 32;\n\tadd.u32 b, %2, 512;\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %4, p1;\n\t"
      "add.u32 a, %1, 40;\n\tadd.u32 b, %2, 640;\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %4, p1;\n\t"
      "add.u32 a, %1, 48;\n\tadd.u32 b, %2, 768;\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %4, p1;\n\t"
      "add.u32 a, %1, 56;\n\tadd.u32 b, %2, 896;\n\tmov.b64 db, {b, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], db, %4, p1;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

}  // namespace tc
}  // namespace rbkv
