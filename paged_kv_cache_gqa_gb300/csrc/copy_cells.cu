// copy_cells: the ordered in-place row mover used by cell compaction.
//
// "KV Cache Design — cells, format, sessions", section 2: a compaction
// changes only cells, so rows move verbatim; an overlapping run is copied
// ascending when it slides down and descending when it slides up, with no
// staging buffer; the moves come in order_moves order.
//
// GB300 design: instead of one row at a time with a barrier after each, a
// move is cut into chunks of min(|dst - src|, len) rows. A chunk's sources and
// destinations never overlap, so all of a chunk's rows, in every pool (all
// layers, K and V), are copied in parallel with 16-byte accesses; a CTA
// barrier separates consecutive chunks, taken in slide order. Consecutive
// moves run in parallel, one CTA per move, as long as none of them writes rows
// another one reads or writes; a move that would starts a new launch. The
// schedule travels in the kernel's parameters (up to 1024 moves per launch),
// so nothing is allocated or copied from the host.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace mtkv {
namespace {

constexpr int kMaxMovesPerLaunch = 1024;
constexpr int kMaxPools = 256;

struct MoveBatch {
  int n_moves;
  int n_pools;
  long long row_bytes;
  mt_move moves[kMaxMovesPerLaunch];
  uint8_t *pools[kMaxPools];
};

template <typename V>
__global__ void __launch_bounds__(256) copy_cells_kernel(const __grid_constant__ MoveBatch b) {
  const mt_move mv = b.moves[blockIdx.x];
  const long long src = mv.src, dst = mv.dst, len = mv.len;
  const long long delta = dst - src;
  const long long chunk = min(delta < 0 ? -delta : delta, len);
  const long long n_chunks = (len + chunk - 1) / chunk;
  const long long vec_per_row = b.row_bytes / (long long)sizeof(V);
  for (long long c = 0; c < n_chunks; ++c) {
    // slide order: descending chunks when moving up, ascending when down
    long long r_lo, r_hi;
    if (delta > 0) {
      r_hi = len - c * chunk;
      r_lo = max(r_hi - chunk, 0LL);
    } else {
      r_lo = c * chunk;
      r_hi = min(r_lo + chunk, len);
    }
    const long long per_pool = (r_hi - r_lo) * vec_per_row;
    const long long total = per_pool * b.n_pools;
    for (long long i = threadIdx.x; i < total; i += blockDim.x) {
      const int pool = (int)(i / per_pool);
      const long long k = i % per_pool;
      const long long row = r_lo + k / vec_per_row;
      const long long v = k % vec_per_row;
      V *base = reinterpret_cast<V *>(b.pools[pool]);
      const V x = base[(src + row) * vec_per_row + v];
      base[(dst + row) * vec_per_row + v] = x;
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace mtkv

using namespace mtkv;

extern "C" mt_status mt_copy_cells(void *const *pools, int n_pools, size_t row_bytes,
                                   int64_t n_cells, const mt_move *moves, int n_moves,
                                   mt_stream stream) {
  if (n_moves < 0 || n_pools < 0 || n_cells < 0)
    return fail(MT_ERR_INVALID_ARG, "mt_copy_cells: negative size");
  if (n_moves == 0 || n_pools == 0) return ok();
  if (!pools || !moves) return fail(MT_ERR_INVALID_ARG, "mt_copy_cells: null pointer");
  if (n_pools > kMaxPools)
    return fail(MT_ERR_UNSUPPORTED, "mt_copy_cells: at most 256 pools per call");
  if (row_bytes == 0 || row_bytes % 4)
    return fail(MT_ERR_INVALID_ARG, "mt_copy_cells: row_bytes must be a positive multiple of 4");
  for (int i = 0; i < n_pools; ++i)
    if (!pools[i] || !aligned16(pools[i]))
      return fail(MT_ERR_INVALID_ARG, "mt_copy_cells: pools must be non-null and 16-byte aligned");
  int bad = -1;
  mt_status st = mt_check_moves(moves, n_moves, n_cells, &bad);
  if (st != MT_OK) return st;  // mt_check_moves set the reason

  std::vector<mt_move> live;
  live.reserve(n_moves);
  for (int i = 0; i < n_moves; ++i)
    if (moves[i].len > 0 && moves[i].src != moves[i].dst) live.push_back(moves[i]);
  if (live.empty()) return ok();

  static thread_local MoveBatch batch;  // 26 KB; kept off the stack
  batch.n_pools = n_pools;
  batch.row_bytes = (long long)row_bytes;
  for (int i = 0; i < n_pools; ++i) batch.pools[i] = static_cast<uint8_t *>(pools[i]);
  const bool v16 = row_bytes % 16 == 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // Moves in one launch run concurrently, so none may write rows another one
  // reads or writes (reading the same source rows is fine).
  struct Run {
    int64_t r0, r1, w0, w1;
  };
  std::vector<Run> runs;
  auto conflicts = [&](const Run &b) {
    for (const Run &a : runs)
      if ((b.w0 < a.r1 && a.r0 < b.w1) || (b.w0 < a.w1 && a.w0 < b.w1) ||
          (a.w0 < b.r1 && b.r0 < a.w1))
        return true;
    return false;
  };
  auto flush = [&]() -> mt_status {
    if (batch.n_moves == 0) return MT_OK;
    if (v16)
      copy_cells_kernel<uint4><<<batch.n_moves, 256, 0, s>>>(batch);
    else
      copy_cells_kernel<uint32_t><<<batch.n_moves, 256, 0, s>>>(batch);
    batch.n_moves = 0;
    runs.clear();
    return cuda_check(cudaGetLastError(), "mt_copy_cells launch");
  };
  batch.n_moves = 0;
  for (const mt_move &m : live) {
    const Run r{m.src, m.src + m.len, m.dst, m.dst + m.len};
    if (batch.n_moves == kMaxMovesPerLaunch || conflicts(r)) {
      st = flush();
      if (st != MT_OK) return st;
    }
    batch.moves[batch.n_moves++] = m;
    runs.push_back(r);
  }
  st = flush();
  return st == MT_OK ? ok() : st;
}
