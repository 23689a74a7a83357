// Shared device helpers for the sm_103a kernels: mbarrier and bulk-copy
// (TMA) wrappers written as inline PTX, bounded waits, and status reporting.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/mtkv.h"

namespace mtkv {

// ---------------------------------------------------------------- status --

__device__ __forceinline__ void report(uint32_t *status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------------------- mbarriers --

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but a warp whose phase is not complete yet is suspended
// (it takes no issue slots) until the phase completes or about `hint_ns`
// nanoseconds have passed.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t *bar, uint32_t parity,
                                                      uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with `parity` to complete. Gives up (returns false)
// when *abort becomes non-zero or after `limit_ns` nanoseconds (checked
// every 8 polls, and never more than 2^31 polls), so no wait can hang.
// After one plain test the waiting warp sleeps in suspended polls of at
// most 20 us each, so a producer or consumer that waits long does not take
// issue slots from the warps it shares a scheduler with.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1; it < 0x80000000u; ++it) {
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if ((it & 7u) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > limit_ns) return false;
    }
  }
  return false;
}

// ---------------------------------------------------- bulk (TMA) copies --

// One contiguous global -> shared copy through the tensor-memory-access
// engine, completing `bytes` of transaction count on `bar`. Both addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Prefetch a contiguous global range into L2 (bytes a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void *g, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(g), "r"(bytes) : "memory");
}

// ------------------------------------------- programmatic dependent launch --
//
// The decode-step kernels are launched with programmatic stream serialisation:
// a kernel may be scheduled while its predecessor in the stream is still
// running, so its launch latency overlaps that kernel's tail. Each such
// kernel first waits until the predecessor has completed and its writes are
// visible (griddepcontrol.wait; a no-op when launched normally), then lets its
// own successor start launching.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The two halves of pdl_enter, for a kernel that does read-only work on its
// inputs (arrays no kernel of this library writes) before it waits: let the
// successor start launching, and (per thread) wait for the predecessor.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Order this thread's earlier generic-proxy global writes before later
// async-proxy (bulk copy / TMA) accesses issued after a barrier.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------------ numerics --

// q8_0 quantisation of one 32-value group, value `x` held by lane `lane` of
// the calling warp (all 32 lanes take part). "KV Cache Design — cells,
// format, sessions", section 3: scale amax/127 in float32, stored as f16;
// code = round-ties-even(x / (amax/127)) clamped to +-127; an all-zero
// group stores scale 0 and codes 0. `blk` is the group's 34-byte block
// {f16 d; int8 q[32]}. The division is IEEE (no fast-math), so any correct
// float32 implementation of the rule gives the same bytes.
__device__ __forceinline__ void q8_quant_group(uint8_t *blk, float x, int lane) {
  float amax = fabsf(x);
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d32 = amax / 127.0f;
  int q = 0;
  if (d32 != 0.0f) {
    // x / d32 through the (IEEE) reciprocal: |t - x/d32| <= |t| 2^-22 <=
    // 3.1e-5 for |t| <= 127, so rounding t gives rint(x / d32) unless t lies
    // within 2^-13 of a half-integer; there the exact division decides
    // (a reciprocal that overflows, for d32 below ~2^-128, takes the exact path)
    const float inv = 1.0f / d32;
    const float t = x * inv;
    const float r = rintf(t);
    q = (int)r;
    if (!isfinite(inv) || fabsf(fabsf(t - r) - 0.5f) < 1.220703125e-4f) q = (int)rintf(x / d32);
    q = max(-127, min(127, q));
  }
  blk[2 + lane] = (uint8_t)(int8_t)q;
  if (lane == 0) *reinterpret_cast<__half *>(blk) = __float2half_rn(d32);
}


__device__ __forceinline__ float2 h2_to_f2(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2 *>(&w);
  return __half22float2(h);
}

// int8 code (two's complement, byte k of w) -> exact float, without the
// integer-to-float conversion unit: place (q + 128) in the low mantissa
// bits of 2^23 and subtract 2^23 + 128.
__device__ __forceinline__ float i8_to_f(uint32_t w_biased, int k) {
  const uint32_t sel = 0x7540u | (uint32_t)k;
  uint32_t bits = __byte_perm(w_biased, 0x4B000000u, sel);
  return __int_as_float((int)bits) - 8388736.0f;
}

}  // namespace mtkv
