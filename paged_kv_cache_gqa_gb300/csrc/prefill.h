// Shared parameters of the multi-query (prefill) kernels: the mma.sync
// kernel (prefill.cu) and the tcgen05 kernel (prefill_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mtkv.h"

namespace mtkv {

constexpr int kMaxPrefillSeqs = 1024;  // sequences per launch (tile offsets in shared memory)

struct PrefillParams {
  const float *q;
  const uint8_t *k_pool;
  const uint8_t *v_pool;
  const int32_t *table;
  const int32_t *ctx;
  const int32_t *q_start;
  const int32_t *spans;
  const int32_t *kv_map;
  float *out;
  float *lse;
  uint32_t *status;
  int B, Hq, Hkv, G, bs, max_blocks;
  int n_tok;  // query rows in q / out (rows outside [0, n_tok) are flagged, not read)
  long long n_phys;
  int row_bytes;
  float qscale;
  // split of each tile's chunks over several CTAs (tcgen05 kernel, when there
  // are fewer tiles than CTAs): per (unit, row) records of D + 4 floats
  // (max, sum, destination row as int bits, unused, unnormalised output),
  // room for rec_units units; rec_hdr[0..1] = (tiles, pieces per tile) of the
  // last launch, for the combine. rec == nullptr: no split.
  float *rec;
  int *rec_hdr;
  int rec_units;
};

// tcgen05 prefill kernel (f16 pools, head_dim 64 or 128, block_size 16 or 32;
// q8_0 and f32 pools of those shapes through staged rows, below).
bool prefill_tc_supported(mt_kv_format fmt, int head_dim, int block_size);

// q8_0 pools on the tcgen05 kernel: the blocks a prefill call reads, staged
// as f16 rows. Block b of sequence s (of the n_seqs sequences of `table`,
// max_blocks entries each) becomes staged block s * max_blocks + b: its bs
// rows of n_kv_heads * head_dim values, value = code * scale rounded once to
// the nearest f16, are written to k16 / v16 (rows of n_kv_heads * head_dim * 2
// bytes), and table16[s][b] = that id; holes, blocks past the context and
// out-of-range ids (flagged in *status) become -1. A staged value beyond the
// f16 range is flagged too (it reads as infinite).
mt_status launch_stage_q8_f16(const uint8_t *k_pool, const uint8_t *v_pool, const int32_t *table,
                              const int32_t *ctx, int n_seqs, int max_blocks, int bs,
                              long long n_phys, int n_kv_heads, int head_dim, int row_bytes,
                              uint8_t *k16, uint8_t *v16, int32_t *table16, uint32_t *status,
                              int n_ctas, cudaStream_t stream);
// f32 pools on the tcgen05 kernel: the blocks a prefill call reads, staged
// as high / low f16 pairs, numbered as launch_stage_q8_f16 numbers them. A
// staged row is the high f16 image of the row's n_kv_heads * head_dim values
// (x rounded to the nearest f16), then the low one (x - high, rounded): rows
// of n_kv_heads * head_dim * 4 bytes in k16 / v16. A value whose high part is
// infinite (outside the f16 range) is flagged in *status.
mt_status launch_stage_f32_pair(const float *k_pool, const float *v_pool, const int32_t *table,
                                const int32_t *ctx, int n_seqs, int max_blocks, int bs,
                                long long n_phys, int n_kv_heads, int head_dim, uint8_t *k16,
                                uint8_t *v16, int32_t *table16, uint32_t *status, int n_ctas,
                                cudaStream_t stream);
// Merge the split pieces' records of the last tcgen05 launch (returns at once
// when it did not split).
mt_status launch_prefill_tc_combine(const PrefillParams &p, int head_dim, int n_ctas,
                                    cudaStream_t stream);
// pair: the pools' rows are high / low f16 images (launch_stage_f32_pair).
mt_status launch_prefill_tc(const PrefillParams &p, int head_dim, int gp, bool pair, int n_ctas,
                            cudaStream_t stream);

}  // namespace mtkv
