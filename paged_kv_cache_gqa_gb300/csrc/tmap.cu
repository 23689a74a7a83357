// Host-side encoding of the pools' tensor maps through the driver's
// cuTensorMapEncodeTiled (looked up once, no link-time driver dependency).
#include <cudaTypedefs.h>

#include <mutex>
#include <string>

#include "internal.h"
#include "tmap.h"

namespace mtkv {
namespace {

mt_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000 *out) {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!fn) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    mt_status st = cuda_check(
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q),
        "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
    if (st != MT_OK) return st;
    if (q != cudaDriverEntryPointSuccess || !f)
      return fail(MT_ERR_CUDA, "driver has no cuTensorMapEncodeTiled");
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  *out = fn;
  return MT_OK;
}

}  // namespace

mt_status encode_pool_map_3d(CUtensorMap *map, const void *pool, long long n_cells, size_t rb,
                             int box_chunks, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  mt_status st = encode_fn(&fn);
  if (st != MT_OK) return st;
  const cuuint64_t dims[3] = {64, (cuuint64_t)(rb / 128), (cuuint64_t)n_cells};
  const cuuint64_t strides[2] = {128, (cuuint64_t)rb};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_chunks, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(pool), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")");
  return MT_OK;
}

mt_status encode_pool_map_words(CUtensorMap *map, const void *pool, long long n_cells, size_t rb,
                                int chunk_bytes, int box_chunks, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  mt_status st = encode_fn(&fn);
  if (st != MT_OK) return st;
  const cuuint64_t dims[3] = {(cuuint64_t)(chunk_bytes / 4), (cuuint64_t)(rb / chunk_bytes),
                              (cuuint64_t)n_cells};
  const cuuint64_t strides[2] = {(cuuint64_t)chunk_bytes, (cuuint64_t)rb};
  const cuuint32_t box[3] = {(cuuint32_t)(chunk_bytes / 4), (cuuint32_t)box_chunks,
                             (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(pool), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")");
  return MT_OK;
}

mt_status encode_out_map_f32(CUtensorMap *map, float *out, long long n_rows, int n_heads,
                             int head_dim, int box_dims, int box_heads, int box_rows) {
  if (box_dims != 32 && box_dims != 16) return fail(MT_ERR_INVALID_ARG, "output box width");
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  mt_status st = encode_fn(&fn);
  if (st != MT_OK) return st;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_heads, (cuuint64_t)n_rows};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 4, (cuuint64_t)n_heads * head_dim * 4};
  const cuuint32_t box[3] = {(cuuint32_t)box_dims, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_dims == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MT_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")");
  return MT_OK;
}

}  // namespace mtkv
