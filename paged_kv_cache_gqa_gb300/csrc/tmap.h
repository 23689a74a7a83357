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

// 3-D tensor map of a pool seen as [cell][chunk of the row][32-bit words]:
// n_cells cells of rb bytes (a multiple of chunk_bytes, which is 16 or 32),
// box = (chunk_bytes / 4, box_chunks, box_rows), no swizzle, zero fill
// outside the tensor. A box wider than the row (box_chunks > rb /
// chunk_bytes) stages each row at a pitch of box_chunks * chunk_bytes
// bytes, the extra chunks zero-filled; the q8_0 decode uses it to place
// staged rows on different shared-memory banks. The pool must be 16-byte
// aligned.
mt_status encode_pool_map_words(CUtensorMap *map, const void *pool, long long n_cells, size_t rb,
                                int chunk_bytes, int box_chunks, int box_rows);

// 3-D tensor map of a float32 output [row][head][dim] (n_rows x n_heads x
// head_dim, rows of n_heads * head_dim floats), box = (box_dims, box_heads,
// box_rows) with box_dims 32 (128-byte swizzle) or 16 (64-byte swizzle):
// the prefill kernel stores a warp's output rows through it. The output
// must be 16-byte aligned and head_dim a multiple of box_dims.
mt_status encode_out_map_f32(CUtensorMap *map, float *out, long long n_rows, int n_heads,
                             int head_dim, int box_dims, int box_heads, int box_rows);

}  // namespace mtkv
