// Host interface of the prefix kernel of the shared-prefix (cascade) decode.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mtkv.h"
#include "cascade.h"

namespace mtkv {

struct PrefixParams {
  const float *q;
  const uint8_t *k_pool;
  const uint8_t *v_pool;
  const int32_t *table;
  const int32_t *ctx;
  const int32_t *spans;
  const int32_t *kv_map;  // [B][MT_KV_MAP_MAX_SPANS][2] (start, len) runs, or null
  uint32_t *status;
  int B, Hq, Hkv, G, bs, max_blocks;
  long long n_phys;
  int row_bytes;
  float qscale;  // softmax scale * log2(e)
  Cascade c;
};

// Whether the prefix kernel is built for this shape (head_dim 64 or 128, and
// 256 for f16 and q8_0 pools; block_size 16 or 32; padded query group <= 8).
bool prefix_supported(mt_kv_format fmt, int head_dim, int block_size, int gp);
// Dynamic shared memory of the prefix kernel for (format, head_dim).
int prefix_smem_bytes(mt_kv_format fmt, int head_dim);
// CTAs of the prefix kernel resident per SM for this head_dim.
int prefix_ctas_per_sm(int head_dim);
mt_status launch_prefix(mt_kv_format fmt, int head_dim, int gp, const PrefixParams &p, int n_ctas,
                        cudaStream_t stream);

}  // namespace mtkv
