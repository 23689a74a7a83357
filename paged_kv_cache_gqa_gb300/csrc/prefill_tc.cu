// Multi-query (prefill) paged attention on the 5th-generation tensor cores
// (tcgen05, tensor-memory accumulators), for f16 pools; q8_0 pools staged as
// f16 rows and f32 pools staged as high / low f16 pairs take the same kernel.
//
// What is computed — exactly what prefill.cu computes (see there): for query
// row i of sequence s at position ctx - n + j, softmax-weighted V over the
// positions t <= its own, t < ctx, not in a hole, inside its window ("Tiered
// KV cache — architecture", sections "The paged-attention block model" and
// "Kernel dispatch"; "KV Cache Design — cells, format, sessions", section 1).
//
// How (GB300): a tile is 128 (query, head) rows of one KV head (one
// tensor-memory lane per row) and the sequence's positions up to the tile's
// last query, in chunks of 128 tokens. CTAs take units round-robin: whole
// tiles, or, when there are fewer tiles than CTAs, pieces of each tile's
// chunks whose unnormalised records a small combine kernel merges. A CTA runs
// three roles that hand work to each other through mbarriers only — no
// CTA-wide barrier inside the chunk loop:
//   * two load warps read the chunk's block ids from the table (a chunk
//     ahead) and stage its K and its V head slices with one tensor copy (TMA,
//     128-byte swizzle) per block and 64-dim half into two rings of stages; a
//     K stage is refilled as soon as its scores are computed, a V stage once
//     its P.V has run (a ring of a single stage, f32 pools at head_dim 128,
//     fills and frees each stage by halves); holes are not read at all;
//   * one MMA warp computes S(c) = Q_hi K^T + Q_lo K^T (paired mode: + Q_hi
//     K_lo^T, K being K_hi + K_lo) (M = 128, N = 128,
//     f16 in, f32 accumulated in tensor memory; q = Q_hi + Q_lo to ~2^-22, so
//     scores keep float32 accuracy; Q read from tensor memory, so only K
//     takes shared-memory bandwidth) into one of two S buffers, as soon as the
//     P.V of the chunk two back (which used that buffer) has run: S(c + 1) is
//     computed while the softmax works on S(c);
//     another computes O += P(c) V(c) once the probabilities of chunk c are
//     in tensor memory (P read from tensor memory, V MN-major straight from
//     its stage), after zeroing the V rows of holes and past the context (P
//     is 0 there but 0 * NaN would not be). The tensor pipe accepts one MMA
//     every ~50 cycles whichever warp issues it, so while one warp waits or
//     commits, the other's MMAs keep it busy;
//   * eight softmax warps, two threads per row (warps w and w + 4 share the
//     tensor-memory lanes 32 (w % 4) .. + 31; each takes 64 of the 128 score
//     columns and half of O): load S, mask it, exchange the row maximum with
//     the partner through shared memory and a two-warp named barrier, run the
//     online softmax, and store f16 probabilities over the scores they came
//     from (each thread over its own columns, already in registers). The
//     output row is rescaled only when the running maximum grows by more than
//     2^8 (probabilities then stay below 256, exact in f16); a tile's output
//     is normalised once at the end.
// The next tile's Q is built during the current tile, a slice of 8 dims per
// chunk, as high / low f16 pairs staged in shared memory (each slice's global
// loads issued at a chunk's start and used at its end); once the last S of a
// tile is complete it is copied into the Q columns of tensor memory, so the
// next tile's first scores are computed while the last chunk's softmax and
// the output of the current tile run.
#include <limits.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "mma.cuh"
#include "prefill.h"
#include "tc.cuh"
#include "tmap.h"

namespace mtkv {
namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kTcRows = 128;       // rows per tile = tensor-memory lanes
constexpr int kTPR = 2;                    // softmax threads per row
constexpr int kSoftWarps = 4 * kTPR;       // warps w, w + 4, ... share lanes 32 (w % 4) ..
constexpr int kLoadWarpK = kSoftWarps;
constexpr int kLoadWarpV = kSoftWarps + 1;
constexpr int kMmaWarpS = kSoftWarps + 2;  // issues S = Q K^T
constexpr int kMmaWarpO = kSoftWarps + 3;  // issues O += P V
constexpr int kTcThreads = 32 * (kSoftWarps + 4);
constexpr int kChunk = 128;                // tokens per chunk
constexpr int kHC = kChunk / kTPR;         // score columns per softmax thread
// tensor-memory columns: S double buffer [0, 128), [128, 256) (S(x) in buffer
// x % 2; P(x) as f16 pairs over the scores it came from: the thread owning
// score columns [kHC h, kHC h + kHC) writes their kHC / 2 probability pairs
// to [kHC h, kHC h + kHC / 2), and in the paired mode the pairs of the low
// parts to [kHC h + kHC / 2, kHC h + kHC)); O [256, 256 + d); the tile's Q as f16 pairs
// (the A operand of S), high [384, 384 + d / 2) and low [448, 448 + d / 2)
constexpr int kSCols = kChunk;
constexpr int kOCol = 2 * kChunk;
constexpr int kQHiCol = 384;
constexpr int kQLoCol = 448;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSplit = 16;       // pieces per tile when tiles are fewer than CTAs

// PAIR: the pools hold each value as a high / low f16 pair (f32 pools,
// staged), so a chunk's K (or V) is two f16 images, high then low.
template <int D, bool PAIR>
struct TcCfg {
  static constexpr int HALVES = D / 64;                 // 64-dim halves of a head
  static constexpr int QSTAGE = D * 512;  // the next tile's Q staged: 128 rows x D x (high, low) f16
  static constexpr int PART = HALVES * kChunk * 128;    // one f16 image of a chunk's K (or V)
  static constexpr int KVB = (PAIR ? 2 : 1) * PART;     // K (or V) of one chunk
  static constexpr int STAGE = 2 * KVB;                 // K and V of one chunk
  static constexpr int STAGES = (D == 64 ? 4 : 2) / (PAIR ? 2 : 1);
  static constexpr int SMEM = 1024 + QSTAGE + STAGES * STAGE;
  // per softmax thread: dims of its part of the row (Q and O), Q slices of 8
  // dims; its warp's region of the Q staging area, and the output box
  // width (dims) of the tensor stores
  static constexpr int DT = D / kTPR;
  static constexpr int NSL = DT / 8;
  static constexpr int REGION = QSTAGE / kSoftWarps;
  static constexpr int CB = DT < 32 ? DT : 32;
  static_assert(REGION >= 2 * NSL * 512 && REGION >= (DT / CB) * 32 * CB * 4, "staging region");
  static_assert(DT >= 16 && (CB == 16 || CB == 32), "output box");
};
static_assert(TcCfg<128, false>::SMEM + 12 * 1024 <= 227 * 1024, "shared memory");
static_assert(TcCfg<64, false>::SMEM + 12 * 1024 <= 227 * 1024, "shared memory");
static_assert(TcCfg<128, true>::SMEM + 12 * 1024 <= 227 * 1024, "shared memory");
static_assert(TcCfg<64, true>::SMEM + 12 * 1024 <= 227 * 1024, "shared memory");

// 2^x by the hardware approximation (relative error ~2^-22, 2^-inf = 0):
// far below the f16 rounding the probabilities get right after.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a + m, b + m) by one packed f32x2 add (each lane rounded as a scalar add).
__device__ __forceinline__ void add2(float a, float b, float m, float &x, float &y) {
  asm("{ .reg .b64 p, q, r; mov.b64 p, {%2, %3}; mov.b64 q, {%4, %4}; add.rn.f32x2 r, p, q; "
      "mov.b64 {%0, %1}, r; }"
      : "=f"(x), "=f"(y)
      : "f"(a), "f"(b), "f"(m));
}

// (s0, s1) += (a, b) by one packed f32x2 add.
__device__ __forceinline__ void acc2(float &s0, float &s1, float a, float b) {
  asm("{ .reg .b64 p, q; mov.b64 p, {%0, %1}; mov.b64 q, {%2, %3}; add.rn.f32x2 p, p, q; "
      "mov.b64 {%0, %1}, p; }"
      : "+f"(s0), "+f"(s1)
      : "f"(a), "f"(b));
}

// One swizzled tensor copy of box (64, 1, rows): 128-byte chunk `chunk` of
// the rows of cells [cell, cell + rows), completing on `bar`.
__device__ __forceinline__ void tma_rows(uint32_t dst, const CUtensorMap *map, int chunk, int cell,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(chunk), "r"(cell), "r"(smem_u32(bar))
      : "memory");
}

// Named barrier of the kTPR warps that share a row quarter (ids 1..4: warps
// w, w + 4, ...) that also ORs a flag.
__device__ __forceinline__ bool pair_vote_or(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.red.or.pred q, %2, %3, p; "
      "selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "n"(32 * kTPR)
      : "memory");
  return r != 0;
}

// The same barrier, ANDing a flag.
__device__ __forceinline__ bool pair_sync_and(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.red.and.pred q, %2, %3, p; "
      "selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "n"(32 * kTPR)
      : "memory");
  return r != 0;
}

struct Tile {
  int s, qt, kvh, n, c, nch;  // sequence, query tile, KV head, queries, context, chunks
};

template <int GP>
__device__ __forceinline__ bool tile_of(const PrefillParams &p, const int *ts, int n_tiles, int t,
                                        Tile &tl) {
  if (t >= n_tiles) return false;
  int lo = 0, hi = p.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ts[mid] <= t) lo = mid; else hi = mid;
  }
  tl.s = lo;
  const int local = t - ts[lo];
  tl.qt = local / p.Hkv;
  tl.kvh = local % p.Hkv;
  tl.n = p.q_start[lo + 1] - p.q_start[lo];
  tl.c = min(max(p.ctx[lo], 0), p.max_blocks * p.bs);
  constexpr int TQ = kTcRows / GP;
  const int last = tl.c - tl.n + min(tl.n, (tl.qt + 1) * TQ) - 1;
  const int reach = min(last + 1, tl.c);
  // at least one chunk, so every tile takes the same hand-offs through all
  // roles (a tile that reaches no position reads nothing and stores zeros)
  tl.nch = reach > 0 ? (reach + kChunk - 1) / kChunk : 1;
  return true;
}

// A unit of work: chunks [cb, ce) of a tile. With n_split pieces per tile,
// unit u is piece u % n_split of tile u / n_split (the tile's chunks cut
// evenly; a piece may be empty when the tile has fewer chunks than pieces).
struct Unit {
  Tile tl;
  int cb, ce;
};

template <int GP>
__device__ __forceinline__ void unit_of(const PrefillParams &p, const int *ts, int n_tiles,
                                        int n_split, int u, Unit &un) {
  tile_of<GP>(p, ts, n_tiles, u / n_split, un.tl);
  const int piece = u % n_split;
  un.cb = piece * un.tl.nch / n_split;
  un.ce = (piece + 1) * un.tl.nch / n_split;
}

// Bits [a, b) of a 64-bit chunk mask (0 <= a, b <= 64).
__device__ __forceinline__ uint64_t bit_range(int a, int b) {
  if (b <= a) return 0ull;
  return (b >= 64 ? ~0ull : ((1ull << b) - 1ull)) & ~((1ull << a) - 1ull);
}

// 8 query values (scaled) as 4 high and 4 low f16 pairs.
__device__ __forceinline__ void split8(const float4 &a, const float4 &b, float qs, uint32_t (&h)[4],
                                       uint32_t (&l)[4]) {
  split_h2(a.x * qs, a.y * qs, h[0], l[0]);
  split_h2(a.z * qs, a.w * qs, h[1], l[1]);
  split_h2(b.x * qs, b.y * qs, h[2], l[2]);
  split_h2(b.z * qs, b.w * qs, h[3], l[3]);
}

// The (query, head) row a softmax thread owns in tile `tl`.
template <int GP>
struct RowOf {
  int j, hg, i;
  bool in, ok;  // in: a query row of this launch; ok: and it has a position
  __device__ __forceinline__ RowOf(const PrefillParams &p, const Tile &tl, int row) {
    constexpr int TQ = kTcRows / GP;
    j = tl.qt * TQ + row / GP;
    hg = row % GP;
    i = p.q_start[tl.s] + j;
    in = j < tl.n && hg < p.G && i >= 0 && i < p.n_tok;
    ok = in && tl.c - tl.n + j >= 0;
  }
};

// W consecutive 32-bit tensor-memory columns of this thread's lane (W a
// multiple of 8).
template <int W>
__device__ __forceinline__ void st_words(uint32_t taddr, const uint32_t (&w)[W]) {
  if constexpr (W % 16 == 0) {
#pragma unroll
    for (int b = 0; b < W; b += 16) tc::st16u(taddr + b, *reinterpret_cast<const uint32_t(*)[16]>(w + b));
  } else {
    static_assert(W == 8, "column count");
    tc::st8u(taddr, w);
  }
}

// Write the row's query as high / low f16 pairs into the Q columns of tensor
// memory (this thread's D / kTPR dims, dims (2c, 2c + 1) in column c of
// each; zeros for rows that hold no query).
template <int D, int GP>
__device__ __forceinline__ void write_q(const PrefillParams &p, const Tile &tl, int row, int hc,
                                        uint32_t q_hi_t, uint32_t q_lo_t) {
  constexpr int DT = D / kTPR, W = DT / 2;
  const RowOf<GP> r(p, tl, row);
  const float *qrow =
      p.q + ((size_t)(r.ok ? r.i : 0) * p.Hq + (size_t)tl.kvh * p.G + r.hg) * D + hc * DT;
  uint32_t h[W], l[W];
#pragma unroll
  for (int j = 0; j < W; j += 4) {  // 8 dims per step
    float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
    if (r.ok) {
      x0 = *reinterpret_cast<const float4 *>(qrow + 2 * j);
      x1 = *reinterpret_cast<const float4 *>(qrow + 2 * j + 4);
    }
    uint32_t hh[4], ll[4];
    split8(x0, x1, p.qscale, hh, ll);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      h[j + t] = hh[t];
      l[j + t] = ll[t];
    }
  }
  st_words<W>(q_hi_t, h);
  st_words<W>(q_lo_t, l);
}

// This thread's DT output values (o, times `mul`; zeros when `zero`) to
// `dst` (null: not stored), by the thread's own 16-byte stores: rows that
// the output's tensor stores do not take (a warp's block of queries that
// runs past its sequence) and the pieces of split tiles.
template <int DT>
__device__ __forceinline__ void store_part(const float (&o)[DT], float mul, bool zero, float *dst) {
  if (!dst) return;
#pragma unroll
  for (int e = 0; e < DT; e += 4)
    *reinterpret_cast<float4 *>(dst + e) =
        zero ? make_float4(0.f, 0.f, 0.f, 0.f)
             : make_float4(o[e] * mul, o[e + 1] * mul, o[e + 2] * mul, o[e + 3] * mul);
}

// One tensor store of box (CB, heads, rows) from shared memory at `src`,
// into the output at (dim x, head y, row z); tracked by this thread's bulk
// group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, int x, int y, int z,
                                             uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Tensor maps of the two pools: [cell][128-byte chunk][64 f16], box (64, 1,
// bs); and, when o_ok, of the output as [row][head][dim], box (CB, G, 32 /
// GP): a block of the (query, head) rows one softmax warp holds.
struct TcMaps {
  CUtensorMap k, v, o;
  int o_ok;
};

// SPLIT: the launch may cut tiles into pieces (records given); without it the
// piece count is the constant 1 and every unit is a whole tile. PAIR: rows of
// the pools are a high f16 image of the values, then a low one (f32 pools,
// staged): S takes Q_lo K_hi and Q_hi K_lo besides Q_hi K_hi, and P.V
// takes P_lo V_hi and P_hi V_lo besides P_hi V_hi.
template <int D, int GP, bool SPLIT, bool PAIR>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ TcMaps maps) {
  using C = TcCfg<D, PAIR>;
  constexpr int ST = C::STAGES;
  // a ring of one stage (PAIR, head_dim 128) fills and frees each stage in
  // two halves with barriers of their own, so half of the next chunk loads
  // while the MMAs read the other: K by 64-dim half (S takes one after the
  // other), V by 64-token half (P.V likewise)
  constexpr int NSB = ST == 1 ? 2 : 1;
  static_assert(NSB == 1 || C::HALVES == 2, "K halves");
  constexpr int R_RUNS = MT_KV_MAP_MAX_SPANS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int ts[kMaxPrefillSeqs + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t k_full[ST * NSB], k_free[ST * NSB], v_full[ST * NSB],
      v_free[ST * NSB], s_full[2],
      p_full[2], pv_done[2], q_full, o_free, drain[2];
  __shared__ uint64_t mask_s[2][ST][2];  // [K / V] staged rows that hold data (not a hole, < ctx)
  __shared__ uint64_t smask_s[2][2];     // the same for the chunk of S(x), by x % 2
  __shared__ float pm_s[2][kTPR][kTcRows];  // partial row maxima: [chunk parity][part][row]
  __shared__ float pl_s[kTPR][kTcRows];     // partial row sums at the tile end
  __shared__ int abort_s;
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *qstage = base;  // the next tile's Q, staged
  uint8_t *ring = base + C::QSTAGE;
  pdl_enter();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // tile offsets: ceil(n_s / TQ) query tiles per sequence, times Hkv
  constexpr int TQ = kTcRows / GP;
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int s = b0 + lane;
      int nt = 0;
      if (s < p.B) {
        const int n = p.q_start[s + 1] - p.q_start[s];
        if (n < 0 || n > max(p.ctx[s], 0)) report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
        nt = n > 0 ? (n + TQ - 1) / TQ * p.Hkv : 0;
      }
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kAll, incl, o);
        if (lane >= o) incl += y;
      }
      if (s < p.B) ts[s] = run + incl - nt;
      run += __shfl_sync(kAll, incl, 31);
    }
    if (lane == 0) ts[p.B] = run;
  }
  if (tid == 0) {
    for (int k = 0; k < ST * NSB; ++k) {
      mbar_init(&k_full[k], 1);
      mbar_init(&k_free[k], 1);
      mbar_init(&v_full[k], 1);
      mbar_init(&v_free[k], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 2);  // the MMAs' commit + the issuing thread (smask_s written)
      mbar_init(&p_full[k], kSoftWarps);
      mbar_init(&pv_done[k], 1);
    }
    mbar_init(&q_full, kSoftWarps);
    mbar_init(&o_free, kSoftWarps);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    abort_s = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int n_tiles = ts[p.B];
  // fewer tiles than CTAs: each tile's chunks are cut into pieces that
  // separate CTAs take, as many as fit in one wave (a second wave of pieces
  // costs more than it saves: 3 pieces of 64 tiles on 152 CTAs ran slower
  // than no split, 2 pieces 1.43x faster); the combine kernel merges them
  int n_split = 1;
  if (SPLIT && n_tiles > 0 && n_tiles < (int)gridDim.x)
    n_split = max(1, min(min((int)gridDim.x / n_tiles, kMaxSplit), p.rec_units / n_tiles));
  const int n_units = n_tiles * n_split;
  if (SPLIT && blockIdx.x == 0 && tid == 0) {
    p.rec_hdr[0] = n_tiles;
    p.rec_hdr[1] = n_split;
  }
  if ((int)blockIdx.x >= n_units) return;
  // the first unit at or after u (same stride as the CTA's) with chunks to run;
  // every role walks the same sequence
  auto live_unit = [&](int &u, Unit &un) -> bool {
    for (; u < n_units; u += gridDim.x) {
      unit_of<GP>(p, ts, n_tiles, n_split, u, un);
      if (un.ce > un.cb) return true;
    }
    return false;
  };
  if (warp == 0) tc::alloc(&tmem_slot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;
  const uint64_t wait_ns = 2000000000ull;
  const int bs_shift = p.bs == 32 ? 5 : 4;
  bool fine = true;  // false once a bounded wait ran out (or another role gave up)

  if (warp == kLoadWarpK || warp == kLoadWarpV) {
    // ================================================================ load
    // one warp stages K, one V: a K stage is refilled as soon as its S has
    // been computed, a V stage once its P.V has run
    const int kv = warp == kLoadWarpV;
    uint64_t *full = kv ? v_full : k_full;
    uint64_t *empty = kv ? v_free : k_free;
    const CUtensorMap *map = kv ? &maps.v : &maps.k;
    const int nb = kChunk >> bs_shift;
    // lane k < 64 / bs reads the table entry of block k of a chunk, one chunk
    // ahead of its use (checked when used)
    auto fetch = [&](const Tile &u, int c) -> int {
      const int pos = c * kChunk + (lane << bs_shift);
      return (lane < nb && pos < u.c) ? p.table[(size_t)u.s * p.max_blocks + (pos >> bs_shift)]
                                      : -1;
    };
    int g = 0;  // chunks staged by this CTA so far (all units)
    int u = blockIdx.x;
    Unit un;
    bool have = live_unit(u, un);
    int raw_next = have ? fetch(un.tl, un.cb) : -1;
    while (have && fine) {
      const Tile &tl = un.tl;
      int u2 = u + (int)gridDim.x;
      Unit nx;
      const bool have_next = live_unit(u2, nx);
      for (int c = un.cb; c < un.ce; ++c, ++g) {
        int phys = raw_next;
        raw_next = c + 1 < un.ce ? fetch(tl, c + 1) : (have_next ? fetch(nx.tl, nx.cb) : -1);
        const int st = g % ST;
        if (phys < -1 || (phys >= 0 && (long long)phys >= p.n_phys)) {
          report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
          phys = -1;
        }
        // rows [a, b) of the chunk hold data (block k = lane)
        const int a = lane << bs_shift, pos = c * kChunk + a;
        const int b = phys >= 0 ? a + min(p.bs, tl.c - pos) : a;
        const uint64_t m0 = bit_range(min(a, 64), min(b, 64));
        const uint64_t m1 = bit_range(max(a - 64, 0), max(b - 64, 0));
        const uint32_t w0 = __reduce_or_sync(kAll, (uint32_t)m0);
        const uint32_t w1 = __reduce_or_sync(kAll, (uint32_t)(m0 >> 32));
        const uint32_t w2 = __reduce_or_sync(kAll, (uint32_t)m1);
        const uint32_t w3 = __reduce_or_sync(kAll, (uint32_t)(m1 >> 32));
        const uint64_t mw0 = ((uint64_t)w1 << 32) | w0, mw1 = ((uint64_t)w3 << 32) | w2;
        // one copy per (block, 64-dim half): lane = k * HALVES + h (PAIR: and
        // one of the low image, Hkv heads further along the row); with two
        // barriers per stage, the copy's half of the stage: its dim half (K)
        // or its token half (V)
        const int k = lane / C::HALVES, h = lane % C::HALVES;
        const int pk = __shfl_sync(kAll, phys, k & 31);
        const int sub = NSB == 1 ? 0 : kv ? (k << bs_shift) >> 6 : h;
        bool waited = true;
#pragma unroll
        for (int j = 0; j < NSB; ++j) {
          uint64_t *fb = &full[st * NSB + j];
          if (g >= ST && !mbar_wait_bounded(&empty[st * NSB + j], (uint32_t)((g / ST) - 1) & 1u,
                                            &abort_s, wait_ns)) {
            // the copies already issued to the stage's first half land first
            for (int j2 = 0; j2 < j; ++j2)
              mbar_wait_bounded(&full[st * NSB + j2], (uint32_t)(g / ST) & 1u, &abort_s, wait_ns);
            waited = false;
            break;
          }
          const bool mine = k < nb && pk >= 0 && sub == j;
          const uint32_t n_copies = __popc(__ballot_sync(kAll, mine));
          if (lane == 0) {
            // the row masks go with the first barrier (K: S reads both
            // before its first MMA); V's token halves each with their own
            if (NSB == 1 || kv == 0) {
              if (j == 0) {
                mask_s[kv][st][0] = mw0;
                mask_s[kv][st][1] = mw1;
              }
            } else {
              mask_s[kv][st][j] = j ? mw1 : mw0;
            }
            mbar_arrive_expect_tx(fb, (n_copies * (PAIR ? 2u : 1u) * 128u) << bs_shift);
          }
          __syncwarp();
          if (mine) {
            const uint32_t dst = smem_u32(ring) +
                                 (uint32_t)(st * C::STAGE + kv * C::KVB + h * (kChunk * 128) +
                                            (k << bs_shift) * 128);
            tma_rows(dst, map, tl.kvh * C::HALVES + h, pk << bs_shift, fb);
            if constexpr (PAIR)
              tma_rows(dst + C::PART, map, (p.Hkv + tl.kvh) * C::HALVES + h, pk << bs_shift, fb);
          }
        }
        if (!waited) {
          fine = false;
          break;
        }
      }
      un = nx;
      u = u2;
      have = have_next;
    }
    // copies still in flight land before the CTA leaves (the last fill of each stage)
    for (int k = 0; k < ST; ++k) {
      if (g <= k) continue;
      const int gl = g - 1 - ((g - 1 - k) % ST);
      for (int j = 0; j < NSB; ++j)
        if (!mbar_wait_bounded(&full[k * NSB + j], (uint32_t)(gl / ST) & 1u, &abort_s, wait_ns))
          fine = false;
    }
  } else if (warp == kMmaWarpS || warp == kMmaWarpO) {
    // ================================================================= MMA
    // two issuing warps share the tensor pipe: while one waits or commits,
    // the other's MMAs keep it busy (one MMA is accepted every ~50 cycles)
    const int role = warp - kMmaWarpS;  // 0: S, 1: P.V
    constexpr uint32_t idesc_s = tc::idesc_f16(kTcRows, kChunk, false);
    constexpr uint32_t idesc_o = tc::idesc_f16(kTcRows, D, true);
    // descriptor bases, advanced per operand by whole 16-byte units
    const uint64_t d_k = tc::desc_sw128(smem_u32(ring), 16, 1024);
    const uint64_t d_v = tc::desc_sw128(smem_u32(ring) + C::KVB, kChunk * 128, 1024);
    int g = 0;
    for (int u = blockIdx.x, k = 0; fine; u += gridDim.x, ++k) {
      Unit un;
      if (!live_unit(u, un)) break;
      // S: this unit's Q is in place
      if (role == 0 && !mbar_wait_bounded(&q_full, (uint32_t)k & 1u, &abort_s, wait_ns)) {
        fine = false;
        break;
      }
      for (int c = un.cb; c < un.ce; ++c) {
        const int x = g + (c - un.cb), st = x % ST;
        if (role == 0) {
          // S(x) = Q_hi K^T + Q_lo K^T into buffer x % 2, once K of chunk x
          // is staged (two barriers per stage: its dim halves one after the
          // other, each freed once its MMAs are done) and P(x - 2) V has run
          // (the softmax has then read S(x - 2) and its row mask, and P(x -
          // 2) is no longer needed)
          if (!mbar_wait_bounded(&k_full[st * NSB], (uint32_t)(x / ST) & 1u, &abort_s, wait_ns) ||
              (x >= 2 && !mbar_wait_bounded(&pv_done[x & 1], (uint32_t)((x - 2) >> 1) & 1u,
                                            &abort_s, wait_ns))) {
            fine = false;
            break;
          }
          const uint64_t kd = tc::desc_advance(d_k, (uint32_t)(st * C::STAGE));
          const uint32_t dcol = tmem + (uint32_t)((x & 1) * kSCols);
          bool staged = true;
#pragma unroll
          for (int j = 0; j < NSB; ++j) {
            if (j > 0 && !mbar_wait_bounded(&k_full[st * NSB + j], (uint32_t)(x / ST) & 1u,
                                            &abort_s, wait_ns)) {
              staged = false;
              break;
            }
            tc::fence_after();
            if (lane == 0) {
              if (j == 0) {
                // the chunk's row mask goes with S(x) (the K stage may be
                // refilled as soon as S(x) is done); published by this
                // thread's arrive below
                smask_s[x & 1][0] = mask_s[0][st][0];
                smask_s[x & 1][1] = mask_s[0][st][1];
              }
#pragma unroll
              for (int hf = j * (C::HALVES / NSB); hf < (j + 1) * (C::HALVES / NSB); ++hf)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  // dims [64 hf + 16 kk, + 16): Q columns 32 hf + 8 kk of each half
                  const uint32_t qc = (uint32_t)(hf * 32 + kk * 8);
                  const uint64_t bd =
                      tc::desc_advance(kd, (uint32_t)(hf * kChunk * 128 + kk * 32));
                  tc::mma_f16_ts(dcol, tmem + kQHiCol + qc, bd, idesc_s, hf + kk > 0);
                  tc::mma_f16_ts(dcol, tmem + kQLoCol + qc, bd, idesc_s, true);
                  if constexpr (PAIR)
                    tc::mma_f16_ts(dcol, tmem + kQHiCol + qc, tc::desc_advance(bd, C::PART),
                                   idesc_s, true);
                }
              if (j == NSB - 1) {
                tc::commit(&s_full[x & 1]);
                tc::commit(&k_free[st * NSB + j]);
                mbar_arrive(&s_full[x & 1]);
              } else {
                tc::commit(&k_free[st * NSB + j]);
              }
            }
            __syncwarp();
          }
          if (!staged) {
            fine = false;
            break;
          }
          continue;
        }
        // P.V: V of chunk x staged (two barriers per stage: its token halves
        // one after the other, each freed once its MMAs are done); its rows
        // without data (holes, past the context) -> 0 first
        uint8_t *vt = ring + (size_t)st * C::STAGE + C::KVB;
        auto zero_rows = [&](int th, uint64_t m) {
          // token half th: u = ((image * HALVES + dim half) * 64 + row) * 8 + 16-byte part
          for (int u = lane; u < C::KVB / 32; u += 32) {
            const int r = (u >> 3) & 63, line = (u >> 9) * kChunk + th * 64 + r;
            if (!((m >> r) & 1ull))
              *reinterpret_cast<uint4 *>(vt + (size_t)line * 128 + (u & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
          }
        };
        bool staged = true;
#pragma unroll
        for (int j = 0; j < NSB; ++j) {
          if (!mbar_wait_bounded(&v_full[st * NSB + j], (uint32_t)(x / ST) & 1u, &abort_s,
                                 wait_ns)) {
            staged = false;
            break;
          }
          bool zeroed = false;
#pragma unroll
          for (int th = j * (2 / NSB); th < (j + 1) * (2 / NSB); ++th) {
            const uint64_t m = mask_s[1][st][th];
            if (m != ~0ull) {
              zero_rows(th, m);
              zeroed = true;
            }
          }
          if (zeroed) {
            tc::fence_proxy_shared();
            __syncwarp();
          }
          // P(x) written; before the tile's first P.V, the previous output read out
          if (j == 0 &&
              (!mbar_wait_bounded(&p_full[x & 1], (uint32_t)(x >> 1) & 1u, &abort_s, wait_ns) ||
               (c == un.cb && k > 0 &&
                !mbar_wait_bounded(&o_free, (uint32_t)(k - 1) & 1u, &abort_s, wait_ns)))) {
            staged = false;
            break;
          }
          tc::fence_after();
          if (lane == 0) {
            // O += P V (P from tensor memory, in S buffer x % 2: tokens
            // [16 kk, 16 kk + 16) at column kHC (kk / J) + 8 (kk % J), J = kHC /
            // 16 K steps per softmax thread's columns; V MN-major: LBO = the
            // distance between its 64-dim halves)
            const uint64_t vd = tc::desc_advance(d_v, (uint32_t)(st * C::STAGE));
            const uint32_t pa = tmem + (uint32_t)((x & 1) * kSCols);
#pragma unroll
            for (int kk = j * (kChunk / 16 / NSB); kk < (j + 1) * (kChunk / 16 / NSB); ++kk) {
              const uint32_t pc = pa + (kk / (kHC / 16)) * kHC + (kk % (kHC / 16)) * 8;
              const uint64_t vk = tc::desc_advance(vd, kk * 2048);
              tc::mma_f16_ts(tmem + kOCol, pc, vk, idesc_o, c > un.cb || kk > 0);
              if constexpr (PAIR) {
                // P_lo: the second half of the thread's columns
                tc::mma_f16_ts(tmem + kOCol, pc + kHC / 2, vk, idesc_o, true);
                tc::mma_f16_ts(tmem + kOCol, pc, tc::desc_advance(vk, C::PART), idesc_o, true);
              }
            }
            if (j == NSB - 1) tc::commit(&pv_done[x & 1]);
            tc::commit(&v_free[st * NSB + j]);
          }
          __syncwarp();
        }
        if (!staged) {
          fine = false;
          break;
        }
      }
      g += un.ce - un.cb;
    }
    // every MMA issued here has completed before tensor memory is released
    if (lane == 0) tc::commit(&drain[role]);
    __syncwarp();
    if (!mbar_wait_bounded(&drain[role], 0, &abort_s, wait_ns)) fine = false;
  } else {
    // ============================================================= softmax
    // thread (row, hc): score columns [HC hc, HC hc + HC) of each chunk, Q
    // and O dims [DT hc, DT hc + DT)
    const int row = tid & (kTcRows - 1), hc = tid >> 7, pair = 1 + (warp & 3);
    const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // lanes of this row
    constexpr int HC = kHC, DT = C::DT;
    constexpr uint64_t kFull = HC == 64 ? ~0ull : (1ull << HC) - 1ull;
    // this warp's region of the Q staging area: the next tile's Q slices of
    // its threads during a tile, its output rows for the tensor stores at the
    // tile's end (one box of 32 rows x CB dims per CB-dim block)
    uint8_t *wreg = qstage + (size_t)warp * C::REGION;
    bool ost_pending = false;  // tensor stores issued from wreg, maybe still reading it
    auto ost_free = [&]() {
      if (ost_pending) {
        if (lane == 0) bulk_wait_read();
        __syncwarp();
        ost_pending = false;
      }
    };
    // this row's record of unit u (split tiles): max, sum, destination, O
    auto record = [&](int u) -> float * {
      return p.rec + ((size_t)u * kTcRows + row) * (D + 4);
    };
    auto dest_of = [&](const Tile &t2) -> int {
      const RowOf<GP> r2(p, t2, row);
      return r2.in ? r2.i * p.Hq + t2.kvh * p.G + r2.hg : -1;
    };
    // pieces of this CTA with no chunks: records that add nothing
    if (n_split > 1) {
      for (int ue = blockIdx.x; ue < n_units; ue += gridDim.x) {
        Unit e;
        unit_of<GP>(p, ts, n_tiles, n_split, ue, e);
        if (e.ce > e.cb) continue;
        float *rr = record(ue);
        for (int d0 = hc * DT; d0 < (hc + 1) * DT; d0 += 4)
          *reinterpret_cast<float4 *>(rr + 4 + d0) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (hc == 0)
          *reinterpret_cast<float4 *>(rr) =
              make_float4(-INFINITY, 0.f, __int_as_float(dest_of(e.tl)), 0.f);
      }
    }
    // this thread's Q columns in tensor memory: high / low pairs at columns
    // kQHiCol / kQLoCol + hc * DT / 2 + [0, DT / 2)
    const uint32_t q_hi_t = t_row + (uint32_t)(kQHiCol + hc * (DT / 2));
    const uint32_t q_lo_t = t_row + (uint32_t)(kQLoCol + hc * (DT / 2));
    int u = blockIdx.x;
    Unit un;
    bool have = live_unit(u, un);
    if (have) {
      write_q<D, GP>(p, un.tl, row, hc, q_hi_t, q_lo_t);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full);
    }
    int g = 0;
    while (have) {
      const Tile &tl = un.tl;
      // the next unit's query rows head for L2 while this unit runs
      int u2 = u + (int)gridDim.x;
      Unit nxu;
      const bool have_next = live_unit(u2, nxu);
      const Tile &nx = nxu.tl;
      const float *qn = nullptr;  // this thread's part of its next-tile query row (or none)
      if (have_next) {
        const RowOf<GP> rn(p, nx, row);
        if (rn.ok) {
          qn = p.q + ((size_t)rn.i * p.Hq + (size_t)nx.kvh * p.G + rn.hg) * D + hc * DT;
#pragma unroll
          for (int e = 0; e < DT; e += 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + e));
        }
      }
      // the next tile's Q, slice k = dims [8k, 8k + 8) of this thread's part
      // of the row, staged in the warp's shared-memory region as 16-byte
      // groups: high pairs in group k, low pairs in group NSL + k (group g of
      // lane l at 512 g + 16 l, so a warp's accesses cover consecutive words)
      constexpr int NSL = C::NSL;
      uint4 *qst = reinterpret_cast<uint4 *>(wreg) + lane;
      auto load_slice = [&](int k, float4 &a, float4 &b) {
        a = b = make_float4(0.f, 0.f, 0.f, 0.f);
        if (qn) {
          a = *reinterpret_cast<const float4 *>(qn + 8 * k);
          b = *reinterpret_cast<const float4 *>(qn + 8 * k + 4);
        }
      };
      auto store_slice = [&](int k, const float4 &a, const float4 &b) {
        uint32_t h[4], l[4];
        split8(a, b, p.qscale, h, l);
        qst[k * 32] = make_uint4(h[0], h[1], h[2], h[3]);
        qst[(NSL + k) * 32] = make_uint4(l[0], l[1], l[2], l[3]);
      };
      const RowOf<GP> rw(p, tl, row);
      if (hc == 0 && rw.j < tl.n && rw.hg < p.G && !rw.in)
        report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
      int lo = 0, hi = rw.ok ? min(tl.c - tl.n + rw.j + 1, tl.c) : 0;
      if (rw.ok && p.spans) {
        lo = max(p.spans[2 * rw.i], 0);
        hi = min(hi, p.spans[2 * rw.i + 1]);
      }
      int ra[R_RUNS], re[R_RUNS];
      if (p.kv_map) {
#pragma unroll
        for (int r = 0; r < R_RUNS; ++r) {
          ra[r] = re[r] = 0;
          if (rw.ok) {
            const int32_t *rp = p.kv_map + ((size_t)rw.i * R_RUNS + r) * 2;
            ra[r] = max(rp[0], 0);
            re[r] = min(rp[0] + rp[1], hi);
          }
        }
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int c = un.cb; c < un.ce; ++c) {
        const int lc = c - un.cb;  // chunk within the unit
        const int x = g + lc;
        const bool last = c + 1 == un.ce;
        // the next unit's Q slice lc: loads in flight across this chunk
        const bool slice = have_next && lc < NSL && !last;
        float4 qa, qb;
        if (slice) load_slice(lc, qa, qb);
        // ---- S(x) complete
        fine = mbar_wait_bounded(&s_full[x & 1], (uint32_t)(x >> 1) & 1u, &abort_s, wait_ns) &&
               fine;
        tc::fence_after();
        if (last && have_next) {
          // every S of this tile is done, so its Q columns are free: the
          // rest of the next tile's Q is staged, then all of it moves into
          // the Q columns
          ost_free();
          for (int k = lc; k < NSL; ++k) {
            float4 a, b;
            load_slice(k, a, b);
            store_slice(k, a, b);
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {  // high, then low
            uint32_t w[DT / 2];
#pragma unroll
            for (int j = 0; j < NSL; ++j) {
              const uint4 gq = qst[(half * NSL + j) * 32];
              w[4 * j] = gq.x;
              w[4 * j + 1] = gq.y;
              w[4 * j + 2] = gq.z;
              w[4 * j + 3] = gq.w;
            }
            st_words<DT / 2>(half ? q_lo_t : q_hi_t, w);
          }
          tc::wait_st();
          tc::fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&q_full);
        }
        // ---- S(x): this thread's HC columns of buffer x % 2 into registers
        const uint32_t s_row = t_row + (uint32_t)((x & 1) * kSCols + hc * HC);
        float sv[HC];
#pragma unroll
        for (int c16 = 0; c16 < HC; c16 += 16) {
          float v[16];
          tc::ld16(s_row + (uint32_t)c16, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) sv[c16 + e] = v[e];
        }
        const uint64_t vm = (smask_s[x & 1][(hc * HC) >> 6] >> ((hc * HC) & 63)) & kFull;
        tc::wait_ld();
        // ---- mask: the row's window, then the staged rows that hold data
        const int pos0 = c * kChunk + hc * HC;  // position of this thread's first column
        uint64_t mk = 0;
        if (p.kv_map) {
#pragma unroll
          for (int r = 0; r < R_RUNS; ++r)
            mk |= bit_range(max(ra[r] - pos0, 0), min(re[r] - pos0, HC));
        } else {
          mk = bit_range(max(lo - pos0, 0), min(hi - pos0, HC));
        }
        mk &= vm;
        // most chunks are wholly readable: only partial ones pay for the mask
        if (mk != kFull) {
#pragma unroll
          for (int h32 = 0; h32 < HC; h32 += 32) {
            const uint32_t m = (uint32_t)(mk >> h32);
#pragma unroll
            for (int e = 0; e < 32; ++e) sv[h32 + e] = (m & (1u << e)) ? sv[h32 + e] : -INFINITY;
          }
        }
        // row maximum: independent chains of 3-input maxima over 16 columns each
        float mq[HC / 16];
#pragma unroll
        for (int j = 0; j < HC / 16; ++j) {
          const float *v = sv + 16 * j;
          float m = max3f(v[0], v[1], v[2]);
#pragma unroll
          for (int e = 3; e < 15; e += 2) m = max3f(m, v[e], v[e + 1]);
          mq[j] = fmaxf(m, v[15]);
        }
        float mown = mq[0];
#pragma unroll
        for (int j = 1; j < HC / 16; ++j) mown = fmaxf(mown, mq[j]);
        // ---- online softmax, rescaling O only when the maximum grows past 2^8.
        // The row's running maximum changes only when one of its scores passes
        // m_run + 8 (or on its first finite score), so the row's parts exchange
        // their maxima only then: one vote of their warps decides (and carries
        // the waits' outcome; a wait that ran out in any part ends the row's
        // loop at the same point)
        const bool grow = mown != -INFINITY && (m_run == -INFINITY || mown > m_run + 8.f);
        if (pair_vote_or(pair, grow || !fine)) {
          pm_s[x & 1][hc][row] = mown;
          if (!pair_sync_and(pair, fine)) {
            fine = false;
            break;
          }
          float mloc = pm_s[x & 1][0][row];
#pragma unroll
          for (int h = 1; h < kTPR; ++h) mloc = fmaxf(mloc, pm_s[x & 1][h][row]);
          const float m_new = fmaxf(m_run, mloc);
          float scale_o = 1.f;
          if (m_new != -INFINITY && (m_run == -INFINITY || m_new > m_run + 8.f)) {
            scale_o = m_run == -INFINITY ? 1.f : exp2f(m_run - m_new);
            l_run *= scale_o;
            m_run = m_new;
          }
          if (c > un.cb && __any_sync(kAll, scale_o != 1.f)) {
            // P(x-1) V has been added to O
            fine = mbar_wait_bounded(&pv_done[(x - 1) & 1], (uint32_t)((x - 1) >> 1) & 1u,
                                     &abort_s, wait_ns) &&
                   fine;
            tc::fence_after();
#pragma unroll 1
            for (int c16 = hc * DT; c16 < (hc + 1) * DT; c16 += 16) {
              float v[16];
              tc::ld16(t_row + kOCol + c16, v);
              tc::wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] *= scale_o;
              tc::st16(t_row + kOCol + c16, v);
            }
            tc::wait_st();
          }
        }
        // ---- probabilities over this thread's own (already loaded) scores
        float ls[4] = {0.f, 0.f, 0.f, 0.f};  // two packed pairs of partial sums
        const float mr = m_run == -INFINITY ? 0.f : m_run;  // all sv are -inf then: p = 0
        const uint32_t p_row = s_row;
        if constexpr (PAIR) {
          // p as high and low f16 (p = high + low to ~2^-22): the high pairs
          // over the first HC / 2 of the thread's columns, the low over the rest
#pragma unroll
          for (int e = 0; e < HC; e += 16) {
            uint32_t h[8], l[8];
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
              float u, w;
              add2(sv[e + 2 * k2], sv[e + 2 * k2 + 1], -mr, u, w);
              const float a = ex2(u), b = ex2(w);
              acc2(ls[2 * (k2 & 1)], ls[2 * (k2 & 1) + 1], a, b);
              split_h2(a, b, h[k2], l[k2]);
            }
            tc::st8u(p_row + (uint32_t)(e / 2), h);
            tc::st8u(p_row + (uint32_t)(HC / 2 + e / 2), l);
          }
        } else {
#pragma unroll
          for (int e = 0; e < HC; e += 32) {
            uint32_t h[16];
#pragma unroll
            for (int k2 = 0; k2 < 16; ++k2) {
              float u, w;
              add2(sv[e + 2 * k2], sv[e + 2 * k2 + 1], -mr, u, w);
              const float a = ex2(u), b = ex2(w);
              acc2(ls[2 * (k2 & 1)], ls[2 * (k2 & 1) + 1], a, b);
              h[k2] = h2_bits(__floats2half2_rn(a, b));
            }
            tc::st16u(p_row + (uint32_t)(e / 2), h);
          }
        }
        l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x & 1]);
        if (slice) {
          ost_free();
          store_slice(lc, qa, qb);
        }
      }
      if (!fine) break;
      const int x_last = g + (un.ce - un.cb) - 1;
      g += un.ce - un.cb;
      // ---- the last P.V, then the normalised row
      fine = mbar_wait_bounded(&pv_done[x_last & 1], (uint32_t)(x_last >> 1) & 1u, &abort_s,
                               wait_ns) &&
             fine;
      tc::fence_after();
      // this thread's part of the output row out of tensor memory (every
      // load in flight, one wait), then O is handed to the next tile's first P.V
      float o[DT];
#pragma unroll
      for (int c16 = 0; c16 < DT; c16 += 16) {
        float v[16];
        tc::ld16(t_row + (uint32_t)(kOCol + hc * DT + c16), v);
#pragma unroll
        for (int e = 0; e < 16; ++e) o[c16 + e] = v[e];
      }
      tc::wait_ld();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free);
      pl_s[hc][row] = l_run;
      if (!pair_sync_and(pair, fine)) {
        fine = false;
        break;
      }
      float l_row = pl_s[0][row];
#pragma unroll
      for (int h = 1; h < kTPR; ++h) l_row += pl_s[h][row];
      if (n_split > 1) {
        // a piece of a split tile: the unnormalised record, merged later
        float *rr = record(u);
        store_part<DT>(o, 1.f, false, rr + 4 + hc * DT);
        if (hc == 0)
          *reinterpret_cast<float4 *>(rr) =
              make_float4(m_run, l_row, __int_as_float(dest_of(tl)), 0.f);
        un = nxu;
        u = u2;
        have = have_next;
        continue;
      }
      const bool any = l_row > 0.f;
      const float inv = any ? 1.f / l_row : 0.f;
      // the warp's 32 rows are QW whole queries of the tile: when all are
      // queries of the sequence, its rows leave by tensor stores from its
      // region, one box of CB dims per block (box row (query, head) = (lane
      // / GP, lane % GP) packed over the G real heads; the 16-byte chunk c of
      // box row k at c ^ (k % 8) for 128-byte rows, c ^ ((k / 2) % 4) for
      // 64-byte rows: the tensor map's swizzle), so the warp moves on
      // without waiting for them
      constexpr int QW = 32 / GP, CB = C::CB, BOX = 32 * CB * 4;
      const int jq0 = tl.qt * TQ + (warp & 3) * QW;
      const int i0 = p.q_start[tl.s] + jq0;  // the warp's first query row
      if (maps.o_ok && jq0 + QW <= tl.n && i0 >= 0 && i0 + QW <= p.n_tok) {
        ost_free();
        const int k = (lane / GP) * p.G + rw.hg;
        const int sw = CB == 32 ? (k & 7) : ((k >> 1) & 3);
        if (rw.hg < p.G) {
#pragma unroll
          for (int j = 0; j < DT / CB; ++j) {
            uint8_t *brow = wreg + j * BOX + k * (CB * 4);
#pragma unroll
            for (int c = 0; c < CB / 4; ++c) {
              const float *v = o + CB * j + 4 * c;
              *reinterpret_cast<float4 *>(brow + ((c ^ sw) << 4)) =
                  any ? make_float4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
        tc::fence_proxy_shared();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < DT / CB; ++j)
            tma_store_3d(&maps.o, hc * DT + CB * j, tl.kvh * p.G, i0, smem_u32(wreg + j * BOX));
          bulk_commit();
        }
        ost_pending = true;
      } else {
        store_part<DT>(
            o, inv, !any,
            rw.in ? p.out + ((size_t)rw.i * p.Hq + (size_t)tl.kvh * p.G + rw.hg) * D + hc * DT
                  : nullptr);
      }
      if (rw.in && p.lse && hc == 0)
        p.lse[(size_t)rw.i * p.Hq + (size_t)tl.kvh * p.G + rw.hg] =
            any ? (m_run + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
      un = nxu;
      u = u2;
      have = have_next;
    }
    // the output's tensor stores land before the CTA (and its shared memory) ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  if (!fine) {
    abort_s = 1;  // the other roles stop waiting within a few polls
    if (lane == 0) report(p.status, MT_STATUS_BIT_TIMEOUT);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

// Merge the pieces of split tiles: one warp per tile row (the grid's warps
// take the launch's tile rows in turn), lane l owns output dims [l D/32,
// (l + 1) D/32); by log-sum-exp over the pieces' (max, sum) records, then
// normalised. A row's headers and the outputs of its first kB pieces are
// all requested before any is used, so a row of up to kB pieces costs one
// L2 round trip. Rows of no query (destination -1) are skipped.
template <int D>
__global__ void __launch_bounds__(256) prefill_tc_combine_kernel(const __grid_constant__ PrefillParams p) {
  constexpr int DV = D / 32, kB = 4;
  pdl_enter();
  const int n_tiles = p.rec_hdr[0], n_split = p.rec_hdr[1];
  if (n_split <= 1) return;
  const int lane = threadIdx.x & 31;
  const size_t pstride = (size_t)kTcRows * (D + 4);  // from one piece of a tile to the next
  const int n_rows = n_tiles * kTcRows;
  for (int w = blockIdx.x * 8 + (threadIdx.x >> 5); w < n_rows; w += gridDim.x * 8) {
    const int t = w / kTcRows, r = w % kTcRows;
    const float *rr = p.rec + ((size_t)t * n_split * kTcRows + r) * (D + 4);
    float m = -INFINITY, l = 0.f;
    int dst = -1;
    if (lane < n_split) {
      const float4 h = __ldcg(reinterpret_cast<const float4 *>(rr + lane * pstride));
      m = h.x;
      l = h.y;
      dst = __float_as_int(h.z);
    }
    // this lane's dims of pieces [j0, j0 + kB)
    float v[kB][DV];
    auto load = [&](int j0) {
#pragma unroll
      for (int jj = 0; jj < kB; ++jj) {
        if (j0 + jj < n_split) {
          const float *op = rr + (j0 + jj) * pstride + 4 + lane * DV;
#pragma unroll
          for (int e = 0; e < DV; e += 2) {
            const float2 x = __ldcg(reinterpret_cast<const float2 *>(op + e));
            v[jj][e] = x.x;
            v[jj][e + 1] = x.y;
          }
        } else {
#pragma unroll
          for (int e = 0; e < DV; ++e) v[jj][e] = 0.f;
        }
      }
    };
    load(0);
    if (!(l > 0.f)) m = -INFINITY;
    float M = m;
    int d = dst;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(kAll, M, o));
      d = max(d, __shfl_xor_sync(kAll, d, o));
    }
    if (d < 0) continue;
    const float f = m == -INFINITY ? 0.f : exp2f(m - M);
    float L = l * f;
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(kAll, L, o);
    float acc[DV];
#pragma unroll
    for (int e = 0; e < DV; ++e) acc[e] = 0.f;
    for (int j0 = 0; j0 < n_split; j0 += kB) {
      if (j0 > 0) load(j0);
#pragma unroll
      for (int jj = 0; jj < kB; ++jj) {
        const float fs = __shfl_sync(kAll, f, (j0 + jj) & 31);
        const float fj = j0 + jj < n_split ? fs : 0.f;  // the same in every lane
        if (fj == 0.f) continue;  // an empty piece (or none): not read into the sum
#pragma unroll
        for (int e = 0; e < DV; ++e) acc[e] = fmaf(fj, v[jj][e], acc[e]);
      }
    }
    const bool any = L > 0.f;
    const float inv = any ? 1.f / L : 0.f;
    float *out = p.out + (size_t)d * D + lane * DV;
#pragma unroll
    for (int e = 0; e < DV; e += 2)
      *reinterpret_cast<float2 *>(out + e) = make_float2(acc[e] * inv, acc[e + 1] * inv);
    if (p.lse && lane == 0)
      p.lse[d] = any ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
  }
}

// q8_0 rows -> f16 rows for the tensor-core prefill. A CTA per (sequence,
// block) unit at a time: the block's bs rows of K and its bs rows of V, each
// contiguous in its pool, arrive in shared memory together by asynchronous
// copies (16 bytes each when the row size allows, else 4), then four
// threads per 32-value group (an f16 scale, then 32 int8 codes, 34 bytes at
// a 2-byte alignment) each convert 8 of its values into 16 bytes of the
// group's 64 bytes of f16 rows, so a warp's stores cover 512 contiguous
// bytes: each value is code * scale rounded once to the nearest f16.
template <int CH>
__device__ __forceinline__ void stage_copy(uint32_t dst, const void *src) {
  if constexpr (CH == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

template <int CH>
__global__ void __launch_bounds__(256) stage_q8_f16_kernel(
    const uint8_t *__restrict__ k_pool, const uint8_t *__restrict__ v_pool,
    const int32_t *__restrict__ table, const int32_t *__restrict__ ctx, int n_seqs,
    int max_blocks, int bs, long long n_phys, int n_groups, int row_bytes,
    uint8_t *__restrict__ k16, uint8_t *__restrict__ v16, int32_t *__restrict__ table16,
    uint32_t *status) {
  extern __shared__ __align__(16) uint8_t raw[];  // bs rows of K, then bs rows of V
  pdl_enter();
  const int tid = threadIdx.x;
  const long long n_units = (long long)n_seqs * max_blocks;
  const size_t rb16 = (size_t)n_groups * 64;
  const int blk_bytes = bs * row_bytes;
  for (long long unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const int s = (int)(unit / max_blocks), b = (int)(unit % max_blocks);
    const int c = max(ctx[s], 0);
    int phys = b * bs < c ? table[unit] : -1;
    if (phys < -1 || (phys >= 0 && (long long)phys >= n_phys)) {
      if (tid == 0) report(status, MT_STATUS_BIT_DEVICE_CHECK);
      phys = -1;
    }
    if (tid == 0) table16[unit] = phys >= 0 ? (int32_t)unit : -1;
    if (phys < 0) continue;
    const int n_valid = min(bs, c - b * bs);  // rows inside the context
    bool big = false;
#pragma unroll 1
    // the block's K rows, then its V rows, all in flight at once
    for (int kv = 0; kv < 2; ++kv) {
      const uint8_t *src = (kv ? v_pool : k_pool) + (size_t)phys * blk_bytes;
      for (int o = tid * CH; o < blk_bytes; o += 256 * CH)
        stage_copy<CH>(smem_u32(raw + kv * blk_bytes + o), src + o);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
#pragma unroll 1
    for (int kv = 0; kv < 2; ++kv) {
      const uint8_t *rows = raw + kv * blk_bytes;
      uint8_t *dst = (kv ? v16 : k16) + (size_t)unit * bs * rb16;
      // quarter q of group g of row r: codes [8q, 8q + 8) -> output bytes
      // [16q, 16q + 16) of the group's 64
      for (int gi = tid; gi < bs * n_groups * 4; gi += 256) {
        const int q = gi & 3, gq = gi >> 2;
        const int r = gq / n_groups, g = gq - r * n_groups;
        const uint16_t *gp = reinterpret_cast<const uint16_t *>(rows + r * row_bytes + g * 34);
        const __half dh = __ushort_as_half(gp[0]);
        const __half2 d2 = __halves2half2(dh, dh);
        // codes exactly as f16 (the bit pattern 0x64XX is 1024 + XX: codes
        // + 128 as bytes, minus 1152), then one f16 multiply by the scale:
        // the exact product rounded to the nearest f16
        const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
          const uint32_t b4 =
              ((uint32_t)gp[2 + 4 * q + j] << 16 | gp[1 + 4 * q + j]) ^ 0x80808080u;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            uint32_t hb = __byte_perm(b4, 0x64646464u, t ? 0x4342 : 0x4140);
            __half2 h = __hsub2(*reinterpret_cast<__half2 *>(&hb), bias);
            h = __hmul2(h, d2);
            w[j + t] = *reinterpret_cast<uint32_t *>(&h);
          }
        }
        // a product rounds to infinity only if |scale| * 128 can reach 65520
        if (r < n_valid && fabsf(__half2float(dh)) * 128.f >= 65504.f) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&w[j]);
            big |= __hisinf(__low2half(h)) || __hisinf(__high2half(h));
          }
        }
        *reinterpret_cast<uint4 *>(dst + (size_t)r * rb16 + (size_t)g * 64 + q * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    __syncthreads();  // the buffer is refilled for the next unit
    if (big) report(status, MT_STATUS_BIT_DEVICE_CHECK);
  }
}

// f32 rows -> high / low f16 rows for the tensor-core prefill: value x
// becomes high = x rounded to the nearest f16 and low = (x - high) rounded
// to the nearest f16 (high + low = x to ~2^-22 relative for |x| inside the
// f16 range; a value whose high part is infinite is flagged). A staged row
// is the high image of the row's hd values, then the low image (hd * 4
// bytes, as the f32 row). A CTA per (sequence, block) unit at a time, each
// thread converting 4 consecutive values per step.
__global__ void __launch_bounds__(256) stage_f32_pair_kernel(
    const float *__restrict__ k_pool, const float *__restrict__ v_pool,
    const int32_t *__restrict__ table, const int32_t *__restrict__ ctx, int n_seqs,
    int max_blocks, int bs, long long n_phys, int hd, uint8_t *__restrict__ k16,
    uint8_t *__restrict__ v16, int32_t *__restrict__ table16, uint32_t *status) {
  pdl_enter();
  const int tid = threadIdx.x, n4 = hd / 4;
  const long long n_units = (long long)n_seqs * max_blocks;
  for (long long unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const int s = (int)(unit / max_blocks), b = (int)(unit % max_blocks);
    const int c = max(ctx[s], 0);
    int phys = b * bs < c ? table[unit] : -1;
    if (phys < -1 || (phys >= 0 && (long long)phys >= n_phys)) {
      if (tid == 0) report(status, MT_STATUS_BIT_DEVICE_CHECK);
      phys = -1;
    }
    if (tid == 0) table16[unit] = phys >= 0 ? (int32_t)unit : -1;
    if (phys < 0) continue;
    const int n_valid = min(bs, c - b * bs);  // rows inside the context
    bool big = false;
#pragma unroll 1
    for (int kv = 0; kv < 2; ++kv) {
      const float4 *src =
          reinterpret_cast<const float4 *>((kv ? v_pool : k_pool) + (size_t)phys * bs * hd);
      uint2 *dst = reinterpret_cast<uint2 *>((kv ? v16 : k16) + (size_t)unit * bs * hd * 4);
      for (int i = tid; i < bs * n4; i += 256) {
        const int r = i / n4, e = i - r * n4;
        const float4 x = __ldg(src + i);
        uint32_t h0, l0, h1, l1;
        split_h2(x.x, x.y, h0, l0);
        split_h2(x.z, x.w, h1, l1);
        uint2 *row = dst + (size_t)r * (hd / 2);  // hd * 4 bytes = hd / 2 eight-byte words
        row[e] = make_uint2(h0, h1);
        row[n4 + e] = make_uint2(l0, l1);
        if (r < n_valid) {
          const __half2 a = *reinterpret_cast<const __half2 *>(&h0);
          const __half2 d = *reinterpret_cast<const __half2 *>(&h1);
          big |= __hisinf(__low2half(a)) || __hisinf(__high2half(a)) ||
                 __hisinf(__low2half(d)) || __hisinf(__high2half(d));
        }
      }
    }
    if (big) report(status, MT_STATUS_BIT_DEVICE_CHECK);
  }
}

template <int D, int GP, bool SPLIT, bool PAIR>
mt_status launch_t(const PrefillParams &p, const TcMaps &m, int n_ctas, cudaStream_t s) {
  auto kern = prefill_tc_kernel<D, GP, SPLIT, PAIR>;
  constexpr int smem = TcCfg<D, PAIR>::SMEM;
  mt_status st = kernel_smem(reinterpret_cast<const void *>(kern), smem,
                             "cudaFuncSetAttribute(prefill tc smem)");
  if (st != MT_OK) return st;
  return cuda_check(launch_pdl(kern, dim3(n_ctas), dim3(kTcThreads), smem, s, p, m),
                    "prefill tc kernel launch");
}

template <int D, bool SPLIT, bool PAIR>
mt_status launch_g(int gp, const PrefillParams &p, const TcMaps &m, int n_ctas, cudaStream_t s) {
  switch (gp) {
    case 1: return launch_t<D, 1, SPLIT, PAIR>(p, m, n_ctas, s);
    case 2: return launch_t<D, 2, SPLIT, PAIR>(p, m, n_ctas, s);
    case 4: return launch_t<D, 4, SPLIT, PAIR>(p, m, n_ctas, s);
    default: return launch_t<D, 8, SPLIT, PAIR>(p, m, n_ctas, s);
  }
}

template <int D, bool PAIR>
mt_status launch_d(int gp, const PrefillParams &p, const TcMaps &m, int n_ctas, cudaStream_t s) {
  return p.rec ? launch_g<D, true, PAIR>(gp, p, m, n_ctas, s)
               : launch_g<D, false, PAIR>(gp, p, m, n_ctas, s);
}

}  // namespace

bool prefill_tc_supported(mt_kv_format fmt, int head_dim, int block_size) {
  return (fmt == MT_KV_F16 || fmt == MT_KV_Q8_0 || fmt == MT_KV_F32) &&
         (head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32);
}

mt_status launch_stage_q8_f16(const uint8_t *k_pool, const uint8_t *v_pool, const int32_t *table,
                              const int32_t *ctx, int n_seqs, int max_blocks, int bs,
                              long long n_phys, int n_kv_heads, int head_dim, int row_bytes,
                              uint8_t *k16, uint8_t *v16, int32_t *table16, uint32_t *status,
                              int n_ctas, cudaStream_t stream) {
  const long long units = (long long)n_seqs * max_blocks;
  if (units == 0) return MT_OK;
  const int grid = (int)std::min<long long>(units, (long long)n_ctas);
  // K and V rows of one block: at most 2 x 32 rows of 8 x 4 x 34 bytes, 68 KB
  const size_t smem = 2 * (size_t)bs * row_bytes;
  auto kern = (row_bytes % 16 == 0) ? stage_q8_f16_kernel<16> : stage_q8_f16_kernel<4>;
  mt_status st = kernel_smem(reinterpret_cast<const void *>(kern), (int)smem,
                             "cudaFuncSetAttribute(q8_0 staging smem)");
  if (st != MT_OK) return st;
  return cuda_check(launch_pdl(kern, dim3(grid), dim3(256), smem, stream, k_pool, v_pool, table,
                               ctx, n_seqs, max_blocks, bs, n_phys, n_kv_heads * head_dim / 32,
                               row_bytes, k16, v16, table16, status),
                    "q8_0 -> f16 staging launch");
}

mt_status launch_stage_f32_pair(const float *k_pool, const float *v_pool, const int32_t *table,
                                const int32_t *ctx, int n_seqs, int max_blocks, int bs,
                                long long n_phys, int n_kv_heads, int head_dim, uint8_t *k16,
                                uint8_t *v16, int32_t *table16, uint32_t *status, int n_ctas,
                                cudaStream_t stream) {
  const long long units = (long long)n_seqs * max_blocks;
  if (units == 0) return MT_OK;
  const int grid = (int)std::min<long long>(units, (long long)n_ctas);
  return cuda_check(launch_pdl(stage_f32_pair_kernel, dim3(grid), dim3(256), 0, stream, k_pool,
                               v_pool, table, ctx, n_seqs, max_blocks, bs, n_phys,
                               n_kv_heads * head_dim, k16, v16, table16, status),
                    "f32 -> high / low f16 staging launch");
}

mt_status launch_prefill_tc_combine(const PrefillParams &p, int head_dim, int n_ctas,
                                    cudaStream_t stream) {
  if (!p.rec) return MT_OK;
  // a split launch has fewer tiles (of 128 rows) than SMs: a warp per row,
  // 8 warps per CTA, 4 CTAs per SM
  auto kern = head_dim == 64 ? prefill_tc_combine_kernel<64> : prefill_tc_combine_kernel<128>;
  return cuda_check(launch_pdl(kern, dim3(4 * n_ctas), dim3(256), 0, stream, p),
                    "prefill tc combine launch");
}

mt_status launch_prefill_tc(const PrefillParams &p, int head_dim, int gp, bool pair, int n_ctas,
                            cudaStream_t stream) {
  // the pools as [cell][128-byte chunk][64 f16] (pair: the chunks of the high
  // image, then those of the low); one copy = bs cells of one chunk
  const long long n_cells = p.n_phys * p.bs;
  TcMaps m;
  mt_status st = encode_pool_map_3d(&m.k, p.k_pool, n_cells, (size_t)p.row_bytes, 1, p.bs);
  if (st != MT_OK) return st;
  st = encode_pool_map_3d(&m.v, p.v_pool, n_cells, (size_t)p.row_bytes, 1, p.bs);
  if (st != MT_OK) return st;
  // the output by tensor stores when it is 16-byte aligned (else every row
  // is stored by the softmax threads themselves)
  m.o_ok = 0;
  if ((reinterpret_cast<uintptr_t>(p.out) & 15u) == 0 && p.n_tok > 0) {
    const int gpe = gp == 1 || gp == 2 || gp == 4 ? gp : 8;  // as launch_g instantiates
    const int cb = std::min(head_dim / kTPR, 32);             // TcCfg<D, PAIR>::CB
    st = encode_out_map_f32(&m.o, p.out, p.n_tok, p.Hq, head_dim, cb, p.G, 32 / gpe);
    if (st != MT_OK) return st;
    m.o_ok = 1;
  }
  if (pair)
    return head_dim == 64 ? launch_d<64, true>(gp, p, m, n_ctas, stream)
                          : launch_d<128, true>(gp, p, m, n_ctas, stream);
  return head_dim == 64 ? launch_d<64, false>(gp, p, m, n_ctas, stream)
                        : launch_d<128, false>(gp, p, m, n_ctas, stream);
}

}  // namespace mtkv
