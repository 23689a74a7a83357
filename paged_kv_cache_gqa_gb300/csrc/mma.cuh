// Warp-level tensor-core helpers (mma.sync.m16n8k16, f16 in, f32
// accumulate) and ldmatrix wrappers shared by the decode and prefix kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace mtkv {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  // not volatile: the compiler may interleave independent MMAs (their only
  // effects are the accumulator registers)
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// high and low f16 halves of a float pair: x ~= hi + lo to ~2^-22 relative
__device__ __forceinline__ void split_h2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  hi = h2_bits(h);
  lo = h2_bits(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
}

// Packed f32x2 arithmetic (one instruction for two lanes, each lane rounded
// exactly as the scalar instruction).
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  float2 r;
  asm("{ .reg .b64 p, q, s; mov.b64 p, {%2, %3}; mov.b64 q, {%4, %5}; add.rn.f32x2 s, p, q; "
      "mov.b64 {%0, %1}, s; }"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
  float2 r;
  asm("{ .reg .b64 p, q, s; mov.b64 p, {%2, %3}; mov.b64 q, {%4, %5}; sub.rn.f32x2 s, p, q; "
      "mov.b64 {%0, %1}, s; }"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  float2 r;
  asm("{ .reg .b64 p, q, s; mov.b64 p, {%2, %3}; mov.b64 q, {%4, %5}; mul.rn.f32x2 s, p, q; "
      "mov.b64 {%0, %1}, s; }"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{ .reg .b64 p, q, t, s; mov.b64 p, {%2, %3}; mov.b64 q, {%4, %5}; mov.b64 t, {%6, %7}; "
      "fma.rn.f32x2 s, p, q, t; mov.b64 {%0, %1}, s; }"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// split_h2 of a float pair with the residual taken by one packed subtraction
__device__ __forceinline__ void split_h2x(float2 x, uint32_t &hi, uint32_t &lo) {
  const __half2 h = __floats2half2_rn(x.x, x.y);
  hi = h2_bits(h);
  const float2 r = f2_sub(x, __half22float2(h));
  lo = h2_bits(__floats2half2_rn(r.x, r.y));
}

}  // namespace mtkv
