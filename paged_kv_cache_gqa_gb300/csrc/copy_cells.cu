// copy_cells: the ordered in-place row mover used by cell compaction.
//
// "KV Cache Design — cells, format, sessions", section 2: a compaction
// changes only cells, so rows move verbatim; an overlapping run is copied
// ascending when it slides down and descending when it slides up, with no
// staging buffer; the moves come in order_moves order.
//
// GB300 design: a run that fits in shared memory (up to 48 KB per pool) moves
// in one round through shared memory with two bulk (TMA) copies, one CTA per
// (move, pool). Longer runs, instead of one row at a time with a barrier after
// each, are cut into chunks of min(|dst - src|, len) rows. A chunk's sources and
// destinations never overlap, so all of a chunk's rows, in every pool (all
// layers, K and V), are copied in parallel with 16-byte accesses; a CTA
// barrier separates consecutive chunks, taken in slide order. Consecutive
// moves run in parallel, one CTA per move, as long as none of them writes rows
// another one reads or writes; a move that would starts a new launch. The
// schedule travels in the kernel's parameters (up to 1024 moves per launch),
// so nothing is allocated or copied from the host.
#include <algorithm>
#include <map>
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
  constexpr int U = 4;  // vectors each thread has in flight per round
  const mt_move mv = b.moves[blockIdx.x];
  const long long src = mv.src, dst = mv.dst, len = mv.len;
  const long long delta = dst - src;
  const long long chunk = min(delta < 0 ? -delta : delta, len);
  const long long n_chunks = (len + chunk - 1) / chunk;
  const long long vec_per_row = b.row_bytes / (long long)sizeof(V);
  // this CTA's share of the pools (blockIdx.y of gridDim.y groups)
  const int p0 = (int)((long long)b.n_pools * blockIdx.y / gridDim.y);
  const int p1 = (int)((long long)b.n_pools * (blockIdx.y + 1) / gridDim.y);
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
    // a chunk's sources and destinations are disjoint: read U vectors, then
    // write them, with no barrier inside the chunk
    const long long per_pool = (r_hi - r_lo) * vec_per_row;
    const long long total = per_pool * (p1 - p0);
    for (long long i0 = threadIdx.x; i0 < total; i0 += (long long)blockDim.x * U) {
      V x[U];
      V *at[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long i = i0 + (long long)u * blockDim.x;
        at[u] = nullptr;
        if (i < total) {
          const int pool = p0 + (int)(i / per_pool);
          const long long k = i % per_pool;
          V *base = reinterpret_cast<V *>(b.pools[pool]);
          const long long off = (r_lo + k / vec_per_row) * vec_per_row + k % vec_per_row;
          x[u] = base[src * vec_per_row + off];
          at[u] = base + dst * vec_per_row + off;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (at[u]) *at[u] = x[u];
    }
    __syncthreads();
  }
}

// A run that fits in shared memory moves in one round: one bulk (TMA) copy
// brings the whole source run of one pool in, and, once it has landed, one
// bulk copy writes it to the destination. Reading everything before writing
// anything gives memmove semantics for any overlap. One CTA per (move, pool).
constexpr int kStagedMax = 48 * 1024;

__global__ void __launch_bounds__(32) copy_cells_staged_kernel(const __grid_constant__ MoveBatch b,
                                                               uint32_t *status) {
  extern __shared__ __align__(128) uint8_t buf[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  const mt_move mv = b.moves[blockIdx.x];
  uint8_t *base = b.pools[blockIdx.y];
  const uint32_t bytes = (uint32_t)(mv.len * b.row_bytes);
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  mbar_arrive_expect_tx(&bar, bytes);
  bulk_g2s(buf, base + mv.src * b.row_bytes, bytes, &bar, policy_evict_first());
  if (!mbar_wait_bounded(&bar, 0, &abort_flag, 2000000000ull)) {
    // nothing is written: report, and let the load land in shared memory
    // (bounded again) before the CTA may retire
    report(status, MT_STATUS_BIT_TIMEOUT);
    mbar_wait_bounded(&bar, 0, &abort_flag, 2000000000ull);
    return;
  }
  asm volatile(
      "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(base + mv.dst * b.row_bytes),
      "r"(smem_u32(buf)), "r"(bytes)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  // the shared-memory source must stay valid until the bulk store has read it
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

}  // namespace
}  // namespace mtkv

using namespace mtkv;

extern "C" mt_status mt_copy_cells(void *const *pools, int n_pools, size_t row_bytes,
                                   int64_t n_cells, const mt_move *moves, int n_moves,
                                   uint32_t *status, mt_stream stream) {
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
  // runs that fit in shared memory (all of them, 16-byte rows) move staged
  bool staged = v16;
  for (const mt_move &m : live)
    if ((long long)m.len * (long long)row_bytes > kStagedMax) staged = false;
  long long batch_max_bytes = 0;
  if (staged) {
    st = kernel_smem(reinterpret_cast<const void *>(copy_cells_staged_kernel), kStagedMax,
                     "cudaFuncSetAttribute(copy_cells staged smem)");
    if (st != MT_OK) return st;
  }

  // Moves in one launch run concurrently, so none may write rows another one
  // reads or writes (reading the same source rows is fine). The launch keeps
  // the union of its read ranges and of its write ranges as sorted disjoint
  // intervals, so each check and insertion is logarithmic.
  struct Union {
    std::map<int64_t, int64_t> iv;  // start -> end, disjoint
    bool hits(int64_t lo, int64_t hi) const {
      auto it = iv.upper_bound(lo);
      if (it != iv.begin() && std::prev(it)->second > lo) return true;
      return it != iv.end() && it->first < hi;
    }
    void add(int64_t lo, int64_t hi) {
      auto it = iv.upper_bound(lo);
      if (it != iv.begin() && std::prev(it)->second >= lo) {
        --it;
        lo = it->first;
        hi = std::max(hi, it->second);
        it = iv.erase(it);
      }
      while (it != iv.end() && it->first <= hi) {
        hi = std::max(hi, it->second);
        it = iv.erase(it);
      }
      iv.emplace(lo, hi);
    }
    void clear() { iv.clear(); }
  };
  Union reads, writes;
  struct Run {
    int64_t r0, r1, w0, w1;
  };
  auto conflicts = [&](const Run &r) {
    return writes.hits(r.w0, r.w1) || reads.hits(r.w0, r.w1) || writes.hits(r.r0, r.r1);
  };
  auto flush = [&]() -> mt_status {
    if (batch.n_moves == 0) return MT_OK;
    if (staged) {
      const dim3 grid((unsigned)batch.n_moves, (unsigned)batch.n_pools);
      copy_cells_staged_kernel<<<grid, 32, (size_t)batch_max_bytes, s>>>(batch, status);
      batch.n_moves = 0;
      reads.clear();
      writes.clear();
      batch_max_bytes = 0;
      return cuda_check(cudaGetLastError(), "mt_copy_cells launch");
    }
    // spread each move's pools over a few CTAs for more parallelism
    const int groups = std::max(1, std::min(batch.n_pools, 2048 / std::max(1, batch.n_moves)));
    const dim3 grid((unsigned)batch.n_moves, (unsigned)std::min(groups, 8));
    if (v16)
      copy_cells_kernel<uint4><<<grid, 256, 0, s>>>(batch);
    else
      copy_cells_kernel<uint32_t><<<grid, 256, 0, s>>>(batch);
    batch.n_moves = 0;
    reads.clear();
    writes.clear();
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
    batch_max_bytes = std::max(batch_max_bytes, (long long)m.len * (long long)row_bytes);
    reads.add(r.r0, r.r1);
    writes.add(r.w0, r.w1);
  }
  st = flush();
  return st == MT_OK ? ok() : st;
}
