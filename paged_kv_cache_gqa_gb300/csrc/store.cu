// KV store: scatter freshly projected float32 rows into their resolved cells,
// converting to the pool's storage format.
//
// "KV Cache Design — cells, format, sessions", section 1 (the store writes
// the cell the allocator resolved, not the position) and section 3 (the one
// store quantiser: q8_0 groups of 32, scale amax/127 kept as f16, codes
// rounded ties-to-even; f16 rounded to nearest even; f32 verbatim).
//
// One warp handles one 32-value group of one row of K or V: lane i loads
// value i (coalesced 128-byte loads), the q8_0 amax is a 5-step shuffle
// reduction (q8_quant_group), and each lane writes its own output element.
#include "common.cuh"
#include "internal.h"

namespace mtkv {
namespace {

template <int FMT>
__global__ void __launch_bounds__(256) kv_store_kernel(uint8_t *__restrict__ k_pool,
                                                       uint8_t *__restrict__ v_pool,
                                                       int64_t n_cells, int row_elems,
                                                       int row_bytes,
                                                       const float *__restrict__ k_new,
                                                       const float *__restrict__ v_new,
                                                       const int64_t *__restrict__ cells,
                                                       int n_rows, uint32_t *status) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int groups = row_elems >> 5;
  const long long warp = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long total = (long long)n_rows * groups;
  if (warp >= total) return;
  const int row = (int)(warp / groups);
  const int g = (int)(warp % groups);
  const bool is_v = blockIdx.y != 0;
  const int64_t cell = cells[row];
  if (cell < 0) return;
  if (cell >= n_cells) {
    if (lane == 0 && !is_v) report(status, MT_STATUS_BIT_DEVICE_CHECK);
    return;
  }
  const float x = (is_v ? v_new : k_new)[(size_t)row * row_elems + g * 32 + lane];
  uint8_t *dst = (is_v ? v_pool : k_pool) + (size_t)cell * row_bytes;
  if (FMT == MT_KV_F32) {
    reinterpret_cast<float *>(dst)[g * 32 + lane] = x;
  } else if (FMT == MT_KV_F16) {
    reinterpret_cast<__half *>(dst)[g * 32 + lane] = __float2half_rn(x);
  } else {
    q8_quant_group(dst + (size_t)g * 34, x, lane);
    // the row is padded to whole 4-byte words: keep the pad bytes zero
    const int pad = row_bytes - groups * 34;
    if (g == groups - 1 && lane < pad) dst[groups * 34 + lane] = 0;
  }
}

}  // namespace
}  // namespace mtkv

using namespace mtkv;

extern "C" mt_status mt_kv_store(mt_kv_format fmt, void *k_pool, void *v_pool, int64_t n_cells,
                                 int n_kv_heads, int head_dim, const float *k_new,
                                 const float *v_new, const int64_t *cells, int n_rows,
                                 uint32_t *status, mt_stream stream) {
  const size_t rb = mt_kv_row_bytes(fmt, n_kv_heads, head_dim);
  if (rb == 0) return fail(MT_ERR_INVALID_ARG, "mt_kv_store: unknown format or bad head shape");
  if (head_dim % 32)
    return fail(MT_ERR_UNSUPPORTED, "mt_kv_store: head_dim must be a multiple of 32");
  if (n_rows < 0 || n_cells < 0)
    return fail(MT_ERR_INVALID_ARG, "mt_kv_store: negative size");
  if (n_rows == 0) return ok();
  if (!k_pool || !v_pool || !k_new || !v_new || !cells)
    return fail(MT_ERR_INVALID_ARG, "mt_kv_store: null pointer");
  if (!aligned16(k_pool) || !aligned16(v_pool))
    return fail(MT_ERR_INVALID_ARG, "mt_kv_store: pools must be 16-byte aligned");
  const int row_elems = n_kv_heads * head_dim;
  const long long warps = (long long)n_rows * (row_elems / 32);
  const long long blocks = (warps + 7) / 8;
  if (blocks > 0x7fffffffLL) return fail(MT_ERR_UNSUPPORTED, "mt_kv_store: too many rows");
  dim3 grid((unsigned)blocks, 2);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto *kp = static_cast<uint8_t *>(k_pool);
  auto *vp = static_cast<uint8_t *>(v_pool);
  cudaError_t e;
  switch (fmt) {
    case MT_KV_F32:
      e = launch_pdl(kv_store_kernel<MT_KV_F32>, grid, dim3(256), 0, s, kp, vp, n_cells, row_elems,
                     (int)rb, k_new, v_new, cells, n_rows, status);
      break;
    case MT_KV_F16:
      e = launch_pdl(kv_store_kernel<MT_KV_F16>, grid, dim3(256), 0, s, kp, vp, n_cells, row_elems,
                     (int)rb, k_new, v_new, cells, n_rows, status);
      break;
    default:
      e = launch_pdl(kv_store_kernel<MT_KV_Q8_0>, grid, dim3(256), 0, s, kp, vp, n_cells, row_elems,
                     (int)rb, k_new, v_new, cells, n_rows, status);
      break;
  }
  mt_status st = cuda_check(e, "mt_kv_store launch");
  return st == MT_OK ? ok() : st;
}
