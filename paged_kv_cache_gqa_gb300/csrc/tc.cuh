// 5th-generation tensor-core helpers (tcgen05, sm_103a) as inline PTX: tensor
// memory allocation, shared-memory matrix descriptors, the kind::f16 MMA with
// its completion signalled on an mbarrier, and tensor-memory loads/stores.
//
// Layout conventions used by the kernels here (checked against a host
// reference on GB300 before use):
//   * operand tiles in shared memory are rows of 128 bytes (64 f16) with the
//     128-byte swizzle: the 16-byte chunk c of row r sits at chunk c ^ (r % 8);
//     8 consecutive rows (1024 bytes) form one swizzle atom;
//   * a K-major operand (K contiguous in each row): SBO = 1024 bytes between
//     8-row groups; a K step of 16 elements advances the start address by 32
//     bytes inside the atom;
//   * an MN-major operand (MN contiguous in each row, rows indexed by K):
//     SBO = 1024 bytes between 8-row (8-K) groups, LBO = the byte distance
//     between 64-element blocks along MN; a K step of 16 advances the start
//     by 2048 bytes;
//   * the f32 accumulator of an M = 128 MMA: row i in tensor-memory lane i,
//     column j at column (base + j); warp w of the CTA reads lanes
//     [32 (w % 4), 32 (w % 4) + 32);
//   * an A operand in tensor memory (M = 128, f16): row i in lane i, column
//     c holding elements (2c, 2c+1), the lower one in the low half.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace mtkv {
namespace tc {

// Allocate `ncols` (a power of two, 32..512) tensor-memory columns; the whole
// warp executes this, and the base address is written to shared memory.
__device__ __forceinline__ void alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Make generic-proxy writes to shared memory (st.shared, cp.async) visible
// to the tensor cores' async proxy (the writer fences, then a barrier).
__device__ __forceinline__ void fence_proxy_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// The descriptor of the operand `bytes` further on: the start address field
// holds address / 16 in 14 bits and every shared address is below 256 KB,
// so the advance never carries out of the field.
__device__ __forceinline__ uint64_t desc_advance(uint64_t d, uint32_t bytes) {
  return d + (uint64_t)(bytes >> 4);
}

// Instruction descriptor of kind::f16: f16 A and B, f32 accumulator, M x N;
// b_mn: B operand MN-major (else K-major); A is K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn) {
  return (1u << 4) | (b_mn ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) = A . B (+ D when acc), issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        bool acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}

// D (tensor memory) = A (tensor memory) . B (+ D when acc): A row i in lane
// i, column c holding its elements (2c, 2c+1), the lower one in the low half;
// a K step of 16 is 8 columns.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, bool acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 16 consecutive f32 columns of this thread's lane.
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

// 4 consecutive 32-bit columns of this thread's lane from raw words.
__device__ __forceinline__ void st4u(uint32_t taddr, uint32_t w0, uint32_t w1, uint32_t w2,
                                     uint32_t w3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(w0),
               "r"(w1), "r"(w2), "r"(w3)
               : "memory");
}

// 8 consecutive 32-bit columns of this thread's lane from raw words.
__device__ __forceinline__ void st8u(uint32_t taddr, const uint32_t (&w)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane from raw words.
__device__ __forceinline__ void st16u(uint32_t taddr, const uint32_t (&w)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}

__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace tc
}  // namespace mtkv
