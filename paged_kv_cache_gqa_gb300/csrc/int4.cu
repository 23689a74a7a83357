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
// One CTA per listed block: pass 1 reduces amax over the block with 16-byte
// loads; pass 2 re-reads the block (now in L2) and writes 8 nibbles (one
// 32-bit word) per thread and step, so every global access is coalesced.
#include "common.cuh"
#include "internal.h"

namespace mtkv {
namespace {

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
  if (threadIdx.x == 0) scales[blockIdx.x] = scale;
  uint32_t *dst = reinterpret_cast<uint32_t *>(nibbles + (size_t)blockIdx.x * (n_elts / 2));
  for (long long i = threadIdx.x; i < n8; i += blockDim.x) {
    float x[8];
    load8<FMT>(src + i * 8 * ES, x);
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      int q = 0;
      if (scale != 0.f) q = max(-8, min(7, (int)rintf(x[e] / scale)));
      word |= (uint32_t)(q + 8) << (4 * e);
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
  if (fmt == MT_KV_F16)
    int4_quant_kernel<MT_KV_F16><<<n_blocks, 256, 0, s>>>(pp, blk_bytes, n_elts, n_phys_blocks,
                                                          blocks, scales, nibbles, status);
  else
    int4_quant_kernel<MT_KV_F32><<<n_blocks, 256, 0, s>>>(pp, blk_bytes, n_elts, n_phys_blocks,
                                                          blocks, scales, nibbles, status);
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
