// Grow-on-demand re-layout of a dense [layer][pos][row] KV store.
//
// "KV cache" (sipllm), section "Design": the store uses its live capacity as
// the per-layer stride, so growing the capacity moves every layer's rows;
// grow_to copies each layer's old rows verbatim from stride old_cap to the
// new stride, which keeps every read bitwise identical to a store
// preallocated at full size.
//
// One 2-D grid: blockIdx.y is the layer, x walks that layer's old_cap rows as
// one contiguous span with 16-byte (or 4-byte) vector copies, four in flight
// per thread.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mtkv {
namespace {

// Each thread keeps U vector loads in flight (all issued before any store):
// with one load per thread the device held too few bytes in flight to cover
// HBM latency (0.67 of the copy peak).
template <typename V, int U>
__global__ void __launch_bounds__(256) relayout_kernel(const uint8_t *__restrict__ src,
                                                       uint8_t *__restrict__ dst,
                                                       long long old_bytes, long long new_bytes) {
  const size_t layer = blockIdx.y;
  const V *__restrict__ s = reinterpret_cast<const V *>(src + layer * old_bytes);
  V *__restrict__ d = reinterpret_cast<V *>(dst + layer * new_bytes);
  const long long n = old_bytes / (long long)sizeof(V);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride * U) {
    V v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i + u * stride < n) v[u] = s[i + u * stride];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i + u * stride < n) d[i + u * stride] = v[u];
  }
}

}  // namespace
}  // namespace mtkv

using namespace mtkv;

extern "C" mt_status mt_kv_relayout(const void *src, void *dst, int n_layers, int64_t old_cap,
                                    int64_t new_cap, size_t row_bytes, mt_stream stream) {
  if (n_layers < 0 || old_cap < 0 || new_cap < old_cap)
    return fail(MT_ERR_INVALID_ARG, "mt_kv_relayout: need 0 <= old_cap <= new_cap");
  if (row_bytes == 0 || row_bytes % 4)
    return fail(MT_ERR_INVALID_ARG, "mt_kv_relayout: row_bytes must be a positive multiple of 4");
  if (n_layers == 0 || old_cap == 0) return ok();
  if (!src || !dst) return fail(MT_ERR_INVALID_ARG, "mt_kv_relayout: null pointer");
  if (!aligned16(src) || !aligned16(dst))
    return fail(MT_ERR_INVALID_ARG, "mt_kv_relayout: buffers must be 16-byte aligned");
  if (n_layers > 65535) return fail(MT_ERR_UNSUPPORTED, "mt_kv_relayout: at most 65535 layers");
  const long long old_bytes = old_cap * (long long)row_bytes;
  const long long new_bytes = new_cap * (long long)row_bytes;
  const bool v16 = row_bytes % 16 == 0;
  const long long n = old_bytes / (v16 ? 16 : 4);
  DeviceInfo di;
  mt_status st = device_info(&di);
  if (st != MT_OK) return st;
  // enough CTAs to cover the device a few times, spread over the layers;
  // each thread copies 4 vectors per round
  long long want = (long long)di.n_sm * 8 / n_layers + 1;
  long long need = (n + 1023) / 1024;
  const unsigned gx = (unsigned)std::max(1LL, std::min(want, need));
  dim3 grid(gx, (unsigned)n_layers);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const auto *sp = static_cast<const uint8_t *>(src);
  auto *dp = static_cast<uint8_t *>(dst);
  if (v16)
    relayout_kernel<uint4, 4><<<grid, 256, 0, s>>>(sp, dp, old_bytes, new_bytes);
  else
    relayout_kernel<uint32_t, 4><<<grid, 256, 0, s>>>(sp, dp, old_bytes, new_bytes);
  st = cuda_check(cudaGetLastError(), "mt_kv_relayout launch");
  return st == MT_OK ? ok() : st;
}
