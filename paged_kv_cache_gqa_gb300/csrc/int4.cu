// Cold-tier int4 codec: per block one float32 scale and packed int4 nibbles.
//
// "Tiered KV cache — architecture", section "The three-tier model": cold
// blocks hold int4-with-scale data, per block a single f32 scale followed by
// ceil(n_elts/2) packed int4 nibbles. Quantiser (the plainest symmetric
// reading): scale = amax/7, q = clamp(rint(x/scale), -8, 7), nibble = q + 8,
// element 2j in the low nibble of byte j; amax == 0 gives scale 0 and every
// nibble 8. Dequantisation writes scale*(nibble-8), rounded to float32 and
// then to the pool's type, into the block the caller assigned (a fresh hot
// id). A block's elements are its cells in pool order [slot][head][dim].
//
// One CTA per listed block: the block (up to 48 KB) arrives in shared memory
// by one bulk (TMA) copy, a block-wide amax reduction follows, then each thread
// packs 8 nibbles (one 32-bit word) per step, so every global access is a bulk
// copy or coalesced; larger blocks take two coalesced passes instead.
#include "common.cuh"
#include "internal.h"

namespace mtkv {
namespace {

// q = clamp(rint(x / scale), -8, 7) with x / scale the IEEE quotient, given
// inv = RN(1 / scale). |x / scale| <= 7, and x * inv is within a few ulp
// (< 2^-19) of the quotient, so rint(x * inv) is the same integer unless the
// product sits within 2^-16 of a half-integer; those rare values take the
// exact division. Bit-identical to dividing every value, at one multiply.
__device__ __forceinline__ int int4_code(float x, float scale, float inv) {
  if (scale == 0.f) return 0;
  const float y = x * inv;
  const float r = rintf(y);
  float q = r;
  // near a half-integer, or no usable reciprocal (a subnormal scale): divide
  if (!(fabsf(y) <= 8.f) || fabsf(fabsf(y - r) - 0.5f) < 1.52587890625e-05f)
    q = rintf(__fdiv_rn(x, scale));
  return max(-8, min(7, (int)q));
}

template <int FMT>
__device__ __forceinline__ void load8(const uint8_t *p, float (&x)[8]) {
  if constexpr (FMT == MT_KV_F16) {
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    float2 f = h2_to_f2(r.x);
    x[0] = f.x; x[1] = f.y;
    f = h2_to_f2(r.y);
    x[2] = f.x; x[3] = f.y;
    f = h2_to_f2(r.z);
    x[4] = f.x; x[5] = f.y;
    f = h2_to_f2(r.w);
    x[6] = f.x; x[7] = f.y;
  } else {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// Packed f32x2 arithmetic: each lane is rounded exactly as the scalar
// instruction would round it (IEEE round-to-nearest-even, subnormals kept).
__device__ __forceinline__ void mul2(float a, float b, float s, float &x, float &y) {
  asm("{ .reg .b64 p, q, r; mov.b64 p, {%2, %3}; mov.b64 q, {%4, %4}; mul.rn.f32x2 r, p, q; "
      "mov.b64 {%0, %1}, r; }"
      : "=f"(x), "=f"(y)
      : "f"(a), "f"(b), "f"(s));
}
__device__ __forceinline__ void add2(float a, float b, float m, float &x, float &y) {
  asm("{ .reg .b64 p, q, r; mov.b64 p, {%2, %3}; mov.b64 q, {%4, %4}; add.rn.f32x2 r, p, q; "
      "mov.b64 {%0, %1}, r; }"
      : "=f"(x), "=f"(y)
      : "f"(a), "f"(b), "f"(m));
}
__device__ __forceinline__ void sub2(float a, float b, float c, float d, float &x, float &y) {
  asm("{ .reg .b64 p, q, r; mov.b64 p, {%2, %3}; mov.b64 q, {%4, %5}; sub.rn.f32x2 r, p, q; "
      "mov.b64 {%0, %1}, r; }"
      : "=f"(x), "=f"(y)
      : "f"(a), "f"(b), "f"(c), "f"(d));
}

// Eight codes packed into one word of nibbles (element e in bits 4e..4e+3).
// t = y + (1.5 * 2^23 + 8) rounds y = x * inv to the nearest integer, ties to
// even (the constant is even and its ulp is 1), and leaves rint(y) + 8 in
// the low 4 bits of t, which is the nibble (|y| <= 7 because |x| <= amax).
// One running maximum of |y - rint(y)| per word catches any value within
// 2^-16 of a half-integer; that word is redone with the exact IEEE division,
// so the result equals clamp(rint(x / scale), -8, 7) + 8 for every element.
// `fast` is false when the reciprocal is not usable (a scale so small that
// 1 / scale overflows), and then every element takes the exact path. The
// products and sums run two elements per instruction, and each pair of
// nibbles becomes a byte with one shift and one bit select.
__device__ __forceinline__ uint32_t int4_pack8(const float (&x)[8], float scale, float inv,
                                               bool fast) {
  if (scale == 0.f) return 0x88888888u;
  constexpr float kMagic8 = 12582920.0f;  // 1.5 * 2^23 + 8
  uint32_t b[4];
  float dev = 0.f;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float y0, y1, t0, t1, r0, r1, d0, d1;
    mul2(x[e], x[e + 1], inv, y0, y1);
    add2(y0, y1, kMagic8, t0, t1);
    add2(t0, t1, -kMagic8, r0, r1);  // rint(y), exactly
    sub2(y0, y1, r0, r1, d0, d1);
    dev = fmaxf(dev, fmaxf(fabsf(d0), fabsf(d1)));
    // low nibble from t0, high nibble from t1 (bits above the byte are
    // dropped by the byte permutes below)
    b[e / 2] = (__float_as_uint(t0) & 0xFu) | ((__float_as_uint(t1) << 4) & ~0xFu);
  }
  uint32_t word = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040),
                              0x5410);
  if (!fast || dev > 0.5f - 1.52587890625e-05f) {
    word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) word |= (uint32_t)(int4_code(x[e], scale, inv) + 8) << (4 * e);
  }
  return word;
}

// Single read: the block arrives in shared memory by one bulk (TMA) copy,
// then 256 threads reduce amax and pack from there. Each CTA holds one block
// (up to 48 KB), so several blocks per SM are in flight at once.
constexpr int kQuantSmemMax = 48 * 1024;

template <int FMT>
__global__ void __launch_bounds__(256) int4_quant_smem_kernel(
    const uint8_t *__restrict__ pool, long long blk_bytes, long long n_elts, long long n_phys,
    const int32_t *__restrict__ blocks, float *__restrict__ scales, uint8_t *__restrict__ nibbles,
    uint32_t *status) {
  constexpr int ES = FMT == MT_KV_F16 ? 2 : 4;
  extern __shared__ __align__(128) uint8_t buf[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ float red[8];
  __shared__ int abort_flag;
  const int id = blocks[blockIdx.x];
  if (id < 0 || id >= n_phys) {
    if (threadIdx.x == 0) report(status, MT_STATUS_BIT_DEVICE_CHECK);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)blk_bytes);
    bulk_g2s(buf, pool + (size_t)id * blk_bytes, (uint32_t)blk_bytes, &bar, policy_evict_first());
  }
  // every thread waits (bounded) for the copy to land
  if (!mbar_wait_bounded(&bar, 0, &abort_flag, 2000000000ull)) {
    if (threadIdx.x == 0) report(status, MT_STATUS_BIT_TIMEOUT);
    return;
  }
  const int n8 = (int)(n_elts / 8);
  float amax = 0.f;
  if constexpr (FMT == MT_KV_F16) {
    // |x| maximum on packed pairs, converted once
    __half2 m2 = __float2half2_rn(0.f);
    for (int i = threadIdx.x; i < n8; i += 256) {
      const uint4 r = *reinterpret_cast<const uint4 *>(buf + (size_t)i * 16);
      m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __half2 *>(&r.x)));
      m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __half2 *>(&r.y)));
      m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __half2 *>(&r.z)));
      m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __half2 *>(&r.w)));
    }
    const float2 mf = __half22float2(m2);
    amax = fmaxf(mf.x, mf.y);
  } else {
    for (int i = threadIdx.x; i < n8; i += 256) {
      float x[8];
      load8<FMT>(buf + (size_t)i * 8 * ES, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax / 7.0f;
  const float inv = scale != 0.f ? 1.0f / scale : 0.f;
  const bool fast = isfinite(inv);
  if (threadIdx.x == 0) scales[blockIdx.x] = scale;
  uint32_t *dst = reinterpret_cast<uint32_t *>(nibbles + (size_t)blockIdx.x * (n_elts / 2));
  for (int i = threadIdx.x; i < n8; i += 256) {
    float x[8];
    load8<FMT>(buf + (size_t)i * 8 * ES, x);
    dst[i] = int4_pack8(x, scale, inv, fast);
  }
}

// Two passes (amax, then quantise with a second read that hits L2), for
// blocks too large for shared memory.
template <int FMT>
__global__ void __launch_bounds__(256) int4_quant_kernel(const uint8_t *__restrict__ pool,
                                                         long long blk_bytes, long long n_elts,
                                                         long long n_phys,
                                                         const int32_t *__restrict__ blocks,
                                                         float *__restrict__ scales,
                                                         uint8_t *__restrict__ nibbles,
                                                         uint32_t *status) {
  constexpr int ES = FMT == MT_KV_F16 ? 2 : 4;
  __shared__ float red[8];
  const int id = blocks[blockIdx.x];
  if (id < 0 || id >= n_phys) {
    if (threadIdx.x == 0) report(status, MT_STATUS_BIT_DEVICE_CHECK);
    return;
  }
  const uint8_t *src = pool + (size_t)id * blk_bytes;
  const long long n8 = n_elts / 8;
  float amax = 0.f;
  for (long long i = threadIdx.x; i < n8; i += blockDim.x) {
    float x[8];
    load8<FMT>(src + i * 8 * ES, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax / 7.0f;
  const float inv = scale != 0.f ? 1.0f / scale : 0.f;
  if (threadIdx.x == 0) scales[blockIdx.x] = scale;
  uint32_t *dst = reinterpret_cast<uint32_t *>(nibbles + (size_t)blockIdx.x * (n_elts / 2));
  for (long long i = threadIdx.x; i < n8; i += blockDim.x) {
    float x[8];
    load8<FMT>(src + i * 8 * ES, x);
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      word |= (uint32_t)(int4_code(x[e], scale, inv) + 8) << (4 * e);
    }
    dst[i] = word;
  }
}

template <int FMT>
__global__ void __launch_bounds__(256) int4_dequant_kernel(uint8_t *__restrict__ pool,
                                                           long long blk_bytes, long long n_elts,
                                                           long long n_phys,
                                                           const int32_t *__restrict__ blocks,
                                                           const float *__restrict__ scales,
                                                           const uint8_t *__restrict__ nibbles,
                                                           uint32_t *status) {
  constexpr int ES = FMT == MT_KV_F16 ? 2 : 4;
  const int id = blocks[blockIdx.x];
  if (id < 0 || id >= n_phys) {
    if (threadIdx.x == 0) report(status, MT_STATUS_BIT_DEVICE_CHECK);
    return;
  }
  uint8_t *dst = pool + (size_t)id * blk_bytes;
  const float scale = scales[blockIdx.x];
  const uint32_t *src = reinterpret_cast<const uint32_t *>(nibbles + (size_t)blockIdx.x * (n_elts / 2));
  const long long n8 = n_elts / 8;
  for (long long i = threadIdx.x; i < n8; i += blockDim.x) {
    const uint32_t word = src[i];
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(scale, (float)((int)((word >> (4 * e)) & 15u) - 8));
    if constexpr (FMT == MT_KV_F16) {
      uint4 r;
      __half2 h;
      h = __halves2half2(__float2half_rn(v[0]), __float2half_rn(v[1]));
      r.x = *reinterpret_cast<uint32_t *>(&h);
      h = __halves2half2(__float2half_rn(v[2]), __float2half_rn(v[3]));
      r.y = *reinterpret_cast<uint32_t *>(&h);
      h = __halves2half2(__float2half_rn(v[4]), __float2half_rn(v[5]));
      r.z = *reinterpret_cast<uint32_t *>(&h);
      h = __halves2half2(__float2half_rn(v[6]), __float2half_rn(v[7]));
      r.w = *reinterpret_cast<uint32_t *>(&h);
      *reinterpret_cast<uint4 *>(dst + i * 8 * ES) = r;
    } else {
      *reinterpret_cast<float4 *>(dst + i * 8 * ES) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4 *>(dst + i * 8 * ES + 16) = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

mt_status check_common(mt_kv_format fmt, const void *pool, int block_size, int n_kv_heads,
                       int head_dim, int64_t n_phys, const void *blocks, int n_blocks,
                       const void *scales, const void *nibbles, const char *who) {
  if (fmt != MT_KV_F16 && fmt != MT_KV_F32)
    return fail(MT_ERR_UNSUPPORTED, std::string(who) + ": cold blocks hold f16 or f32 pools");
  if (block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0 || n_phys < 0 || n_blocks < 0)
    return fail(MT_ERR_INVALID_ARG, std::string(who) + ": bad sizes");
  if (((long long)n_kv_heads * head_dim) % 8)
    return fail(MT_ERR_UNSUPPORTED, std::string(who) + ": n_kv_heads*head_dim must be a multiple of 8");
  if (n_blocks && (!pool || !blocks || !scales || !nibbles))
    return fail(MT_ERR_INVALID_ARG, std::string(who) + ": null pointer");
  if (n_blocks && (!aligned16(pool) || !aligned16(nibbles)))
    return fail(MT_ERR_INVALID_ARG, std::string(who) + ": pool and nibbles must be 16-byte aligned");
  return MT_OK;
}

}  // namespace
}  // namespace mtkv

using namespace mtkv;

extern "C" mt_status mt_kv_quant_int4(mt_kv_format fmt, const void *pool, int block_size,
                                      int n_kv_heads, int head_dim, int64_t n_phys_blocks,
                                      const int32_t *blocks, int n_blocks, float *scales,
                                      uint8_t *nibbles, uint32_t *status, mt_stream stream) {
  mt_status st = check_common(fmt, pool, block_size, n_kv_heads, head_dim, n_phys_blocks, blocks,
                              n_blocks, scales, nibbles, "mt_kv_quant_int4");
  if (st != MT_OK) return st;
  if (n_blocks == 0) return ok();
  const long long n_elts = (long long)block_size * n_kv_heads * head_dim;
  const long long blk_bytes = (long long)mt_kv_row_bytes(fmt, n_kv_heads, head_dim) * block_size;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const auto *pp = static_cast<const uint8_t *>(pool);
  if (blk_bytes <= kQuantSmemMax && blk_bytes % 16 == 0) {
    if (fmt == MT_KV_F16) {
      mt_status st = kernel_smem(reinterpret_cast<const void *>(int4_quant_smem_kernel<MT_KV_F16>),
                                 kQuantSmemMax, "cudaFuncSetAttribute(int4 quant smem)");
      if (st != MT_OK) return st;
      int4_quant_smem_kernel<MT_KV_F16><<<n_blocks, 256, (size_t)blk_bytes, s>>>(
          pp, blk_bytes, n_elts, n_phys_blocks, blocks, scales, nibbles, status);
    } else {
      mt_status st = kernel_smem(reinterpret_cast<const void *>(int4_quant_smem_kernel<MT_KV_F32>),
                                 kQuantSmemMax, "cudaFuncSetAttribute(int4 quant smem)");
      if (st != MT_OK) return st;
      int4_quant_smem_kernel<MT_KV_F32><<<n_blocks, 256, (size_t)blk_bytes, s>>>(
          pp, blk_bytes, n_elts, n_phys_blocks, blocks, scales, nibbles, status);
    }
  } else if (fmt == MT_KV_F16) {
    int4_quant_kernel<MT_KV_F16><<<n_blocks, 256, 0, s>>>(pp, blk_bytes, n_elts, n_phys_blocks,
                                                          blocks, scales, nibbles, status);
  } else {
    int4_quant_kernel<MT_KV_F32><<<n_blocks, 256, 0, s>>>(pp, blk_bytes, n_elts, n_phys_blocks,
                                                          blocks, scales, nibbles, status);
  }
  st = cuda_check(cudaGetLastError(), "mt_kv_quant_int4 launch");
  return st == MT_OK ? ok() : st;
}

extern "C" mt_status mt_kv_dequant_int4(mt_kv_format fmt, void *pool, int block_size,
                                        int n_kv_heads, int head_dim, int64_t n_phys_blocks,
                                        const int32_t *dst_blocks, int n_blocks,
                                        const float *scales, const uint8_t *nibbles,
                                        uint32_t *status, mt_stream stream) {
  mt_status st = check_common(fmt, pool, block_size, n_kv_heads, head_dim, n_phys_blocks,
                              dst_blocks, n_blocks, scales, nibbles, "mt_kv_dequant_int4");
  if (st != MT_OK) return st;
  if (n_blocks == 0) return ok();
  const long long n_elts = (long long)block_size * n_kv_heads * head_dim;
  const long long blk_bytes = (long long)mt_kv_row_bytes(fmt, n_kv_heads, head_dim) * block_size;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto *pp = static_cast<uint8_t *>(pool);
  if (fmt == MT_KV_F16)
    int4_dequant_kernel<MT_KV_F16><<<n_blocks, 256, 0, s>>>(pp, blk_bytes, n_elts, n_phys_blocks,
                                                            dst_blocks, scales, nibbles, status);
  else
    int4_dequant_kernel<MT_KV_F32><<<n_blocks, 256, 0, s>>>(pp, blk_bytes, n_elts, n_phys_blocks,
                                                            dst_blocks, scales, nibbles, status);
  st = cuda_check(cudaGetLastError(), "mt_kv_dequant_int4 launch");
  return st == MT_OK ? ok() : st;
}
