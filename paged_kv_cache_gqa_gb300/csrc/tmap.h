// Tensor maps (TMA descriptors) of the KV pools, encoded on the host.
#pragma once

#include <cuda.h>
#include <stddef.h>

#include "../../include/mtkv.h"

namespace mtkv {

// 3-D tensor map of an f16 pool seen as [cell][128-byte chunk of the row][64
// f16]: n_cells cells of rb bytes (rb a multiple of 128), box = (64,
// box_chunks, box_rows), 128-byte swizzle, zero fill outside the tensor. The
// pool must be 16-byte aligned.
mt_status encode_pool_map_3d(CUtensorMap *map, const void *pool, long long n_cells, size_t rb,
                             int box_chunks, int box_rows);

}  // namespace mtkv
