// Fifth-generation tensor core helpers (sm_100 family): tensor memory
// allocation, shared-memory matrix descriptors, tcgen05.mma with fp32
// accumulators in TMEM, commit to an mbarrier, and TMEM -> register loads.
//
// Operand layout used throughout: "K-major, 128-byte swizzle".  A tile of R
// rows (the M or N side) by 128 columns (the K side) of a 16-bit type is
// stored as two 64-column halves, each R rows x 128 bytes; inside a half, the
// 16-byte chunk c of row r sits at chunk c ^ (r % 8) (the pattern a 2-D TMA
// load with 128-byte swizzle produces; swz_tma() computes the address).
// Eight rows form a 1024-byte atom, so the descriptor's stride between 8-row
// groups is 1024 bytes; a K step of 16 elements advances the start address
// by 32 bytes inside a half, and the next half starts R * 128 bytes later.
#pragma once

#include "msa_device.cuh"

namespace msa {

// Warp-wide: allocate `ncols` TMEM columns (power of two >= 32); the base
// address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
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

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 1024-byte
// stride between 8-row groups; `saddr` is a shared-window byte address.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// As sdesc_sw128 with another stride between 8-row groups (a multiple of 16).
__device__ __forceinline__ uint64_t sdesc_sw128_sbo(uint32_t saddr, uint32_t sbo_bytes) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
         ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);
}

// Descriptor of an MN-major operand with 128-byte swizzle: 64-element (128 B)
// rows of the MN dimension, 8 rows of K per 1 KB atom; lbo_bytes between the
// 64-element MN blocks, 1 KB between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo_bytes) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16 with fp32 accumulation, both operands
// K-major.  fmt: 0 = fp16, 1 = bf16 (A and B must share it).
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t fmt, uint32_t M, uint32_t N) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
// As idesc_f16 with B MN-major (bit 16).
__host__ __device__ constexpr uint32_t idesc_f16_bmn(uint32_t fmt, uint32_t M, uint32_t N) {
  return idesc_f16(fmt, M, N) | (1u << 16);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K step; issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Lean forms for an issuing loop: a shared-memory descriptor passed as its two
// 32-bit words, so that a K step (which only moves the 14-bit start-address
// field in the low word; shared-window addresses stay below 2^18 bytes, so
// the field never carries) costs one integer add; the accumulate flag is a
// compile-time constant.
template <bool kAcc>
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint32_t alo, uint32_t ahi,
                                        uint32_t blo, uint32_t bhi, uint32_t idesc) {
  asm volatile(
      "{\n .reg .b64 a, b;\n .reg .pred p;\n mov.b64 a, {%1, %2};\n mov.b64 b, {%3, %4};\n"
      " setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n}" ::"r"(d_tmem),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "n"(kAcc ? 1 : 0)
      : "memory");
}
// A operand in TMEM: M rows = TMEM lanes, each 32-bit column holding two
// consecutive K elements (lower half first); one K step of 16 elements spans
// 8 columns from a_tmem.
template <bool kAcc>
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t blo,
                                        uint32_t bhi, uint32_t idesc) {
  asm volatile(
      "{\n .reg .b64 b;\n .reg .pred p;\n mov.b64 b, {%2, %3};\n setp.ne.b32 p, %5, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "n"(kAcc ? 1 : 0)
      : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Warp-wide: thread i receives TMEM lane (lane base of taddr) + i, 32
// consecutive 32-bit columns starting at the column of taddr.  A warp may only
// address the 32-lane quarter (warp id % 4) of TMEM.  Complete with
// tmem_ld_wait() before reading the registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// As tmem_ld32 for 64 consecutive columns.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr)
               : "memory");
}
// As tmem_ld32 for 4 consecutive columns.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Warp-wide: thread i writes 32 consecutive 32-bit columns of TMEM lane (lane
// base of taddr) + i.  Complete with tmem_st_wait() before signalling a reader.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk c (0..15) of row r in a K-major SW128 tile of
// `rows` rows (two 64-column halves of rows * 128 bytes).
__device__ __forceinline__ uint32_t kmaj_off(int r, int c, int rows) {
  return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Descriptor of K step ks (16 elements) of a K-major SW128 tile at `base`.
__device__ __forceinline__ uint64_t kstep_desc(uint32_t base, int ks, int rows) {
  return sdesc_sw128(base + (uint32_t)((ks >> 2) * rows * 128 + (ks & 3) * 32));
}

}  // namespace msa
