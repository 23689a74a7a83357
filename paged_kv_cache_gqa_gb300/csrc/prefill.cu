// Multi-query (prefill) paged attention, for sm_103a.
//
// What is computed — for every query row i of sequence s (rows q_start[s] ..
// q_start[s+1]-1, n of them) and query head h: query j = i - q_start[s] sits
// at position ctx - n + j and attends to the positions t <= its own, t < ctx,
// whose block is not a hole ("Tiered KV cache — architecture", sections "The
// paged-attention block model" and "Kernel dispatch": context and query
// lengths per sequence, kInvalidBlockId logits are -infinity), within its
// window: one [lo, hi) pair or up to MT_KV_MAP_MAX_SPANS (start, len) runs
// ("KV Cache Design — cells, format, sessions", section 1: the three window
// modes, read as logical positions). out = softmax-weighted V, lse = the
// natural log-sum-exp of the scaled logits.
//
// Which kernel: head_dim 64 and 128 run the tcgen05 kernel (prefill_tc.cu) —
// f16 pools directly, q8_0 pools after a pass that stages the call's blocks
// as f16 rows, f32 pools after one that stages them as high / low f16 pairs.
// The kernel below takes head_dim 256 (f16, q8_0).
//
// How (GB300): a tile is 64 rows (query token, head) of one KV head — 64/GP
// consecutive queries of one sequence times the GP (padded) heads of the
// group — and every block of the sequence up to the tile's last position.
// CTAs take whole tiles round-robin, so every output is written once,
// normalised, with no split-K combine. The block ring, the f16 tiles and the
// per-warp tensor-core math are the multi-query core (mq.cuh): each staged
// block serves all 64 rows. The next unit's block id is loaded one iteration
// ahead, so no global load sits between a stage's release and its next copy.
#include <limits.h>
#include <math.h>

#include <algorithm>
#include <string>

#include "common.cuh"
#include "internal.h"
#include "mq.cuh"
#include "prefill.h"

namespace mtkv {
namespace {

constexpr uint64_t kPrefillWsBytes = 256;
// Records for tiles split over several CTAs (tcgen05 kernel): room for
// 2 x kSplitCtas units, enough whenever the grid has at most kSplitCtas CTAs
// (the kernel splits only while tiles are fewer than CTAs).
constexpr int kSplitCtas = 160;

// q8_0 and f32 pools on the tcgen05 kernel: the call's blocks staged as f16
// rows (launch_stage_q8_f16) or high / low f16 rows (launch_stage_f32_pair):
// a table of n_seqs x max_blocks staged ids, then the K and the V staged
// pools of n_seqs x max_blocks x block_size rows (2 or 4 bytes per value). 0
// when the call does not stage (f16 pools, other shapes; staged ids that
// would not fit the kernel's 32-bit cell indices: the call is refused).
size_t tc_stage_bytes(const mt_paged_prefill_args *a) {
  if (a->fmt == MT_KV_F16 || !prefill_tc_supported(a->fmt, a->head_dim, a->block_size)) return 0;
  const long long cells = (long long)a->n_seqs * a->max_blocks * a->block_size;
  if (cells <= 0 || cells >= (1LL << 31)) return 0;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  const size_t vb = a->fmt == MT_KV_F32 ? 4 : 2;
  return up((size_t)a->n_seqs * a->max_blocks * 4) +
         2 * up((size_t)cells * a->n_kv_heads * a->head_dim * vb);
}

// Bytes of split records a call may need: 0 unless the tensor-core kernel
// runs and the query count leaves fewer tiles than kSplitCtas (every sequence
// has at least ceil(n_s / TQ) tiles per KV head, so the tile count is at
// least Hkv * ceil(n_tokens / TQ)).
size_t prefill_rec_bytes(const mt_paged_prefill_args *a, int GP) {
  if (!prefill_tc_supported(a->fmt, a->head_dim, a->block_size) || GP == 0) return 0;
  const long long TQ = 128 / GP;
  const long long min_tiles = (long long)a->n_kv_heads * ((a->n_tokens + TQ - 1) / TQ);
  if (min_tiles >= kSplitCtas) return 0;
  return (size_t)2 * kSplitCtas * 128 * (a->head_dim + 4) * sizeof(float);
}

// The CTA's walk over its tiles (blockIdx.x, + gridDim.x, ...) and their
// blocks [0, nb). A tile whose rows read nothing still has one (empty) unit,
// so its outputs are written.
template <int GP>
struct PIter {
  int tile, s, qt, kvh, nb, b, n, c;
  __device__ __forceinline__ void start(const PrefillParams &p, const int *ts, int n_tiles,
                                        int t) {
    tile = t < n_tiles ? t : -1;
    b = 0;
    if (tile < 0) return;
    int lo = 0, hi = p.B;  // last s with ts[s] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ts[mid] <= t) lo = mid; else hi = mid;
    }
    s = lo;
    const int local = t - ts[s];
    qt = local / p.Hkv;
    kvh = local % p.Hkv;
    n = p.q_start[s + 1] - p.q_start[s];
    const int cmax = p.max_blocks * p.bs;
    c = min(max(p.ctx[s], 0), cmax);
    constexpr int TQ = mq::kRows / GP;
    const int last = c - n + min(n, (qt + 1) * TQ) - 1;  // position of the tile's last query
    const int reach = min(last + 1, c);
    nb = reach > 0 ? (reach + p.bs - 1) / p.bs : 1;
  }
  __device__ __forceinline__ void next(const PrefillParams &p, const int *ts, int n_tiles) {
    if (++b < nb) return;
    start(p, ts, n_tiles, tile + (int)gridDim.x);
  }
};

// Block id of the iterator's unit, -1 for holes, flagged ids, units past the
// sequence's context and walks past the last tile.
template <int GP>
__device__ __forceinline__ int unit_phys(const PrefillParams &p, const PIter<GP> &it) {
  if (it.tile < 0 || it.b * p.bs >= it.c) return -1;
  const int phys = p.table[(size_t)it.s * p.max_blocks + it.b];
  if (phys == MT_INVALID_BLOCK_ID) return -1;
  if (phys < 0 || (long long)phys >= p.n_phys) {
    if (threadIdx.x == 0) report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
    return -1;
  }
  return phys;
}

template <int FMT, int D, int GP>
__global__ void __launch_bounds__(mq::kThreads, 2)
    prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = mq::Cfg<FMT, D>;
  using mq::kAll;
  constexpr int TQ = mq::kRows / GP;
  constexpr int S = C::STAGES;
  constexpr int R_RUNS = MT_KV_MAP_MAX_SPANS;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  uint8_t *tiles = smem + S * C::RAW_STAGE;
  float *scales = reinterpret_cast<float *>(tiles + C::TILE_BYTES);
  __shared__ int ts[kMaxPrefillSeqs + 1];           // first tile of each sequence
  __shared__ int phys_ring[S];                       // block id staged in each slot
  __shared__ int win_s[2 * mq::kWarps];
  __shared__ int2 runs_s[mq::kRows][R_RUNS];        // kv_map runs of the tile's rows
  pdl_enter();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, c4 = lane & 3;
  const int bs = p.bs;

  // tile offsets: ceil(n_s / TQ) query tiles per sequence, times Hkv
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int s = base + lane;
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
  __syncthreads();
  const int n_tiles = ts[p.B];
  if ((int)blockIdx.x >= n_tiles) return;

  PIter<GP> cur, ahead;
  cur.start(p, ts, n_tiles, blockIdx.x);
  ahead = cur;
  int ahead_phys = unit_phys(p, ahead);
#pragma unroll
  for (int i = 0; i < S - 1; ++i) {
    mq::issue_block<FMT, D>(p.k_pool, p.v_pool, p.row_bytes, bs, ahead.kvh, ahead_phys, ring, i);
    if (threadIdx.x == 0) phys_ring[i] = ahead_phys;
    if (ahead.tile >= 0) ahead.next(p, ts, n_tiles);
    ahead_phys = unit_phys(p, ahead);
  }

  mq::Rows<D> st;
  if constexpr (C::QS) st.qs = smem_u32(smem + C::SMEM - C::QS_BYTES) + warp * C::QS_WARP;
  int lo_r[2] = {0, 0}, hi_r[2] = {0, 0};  // each row's window bounds (causal, ctx included)
  int orow[2] = {-1, -1};                  // (query row * Hq + head), -1: padding row
  int ulo = 0, uhi = 0;                    // union of the tile's windows
  const bool use_map = p.kv_map != nullptr;

  auto flush = [&]() {
    const float2 l = mq::row_sums(st);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      if (orow[half] < 0) continue;
      const float lh = half ? l.y : l.x;
      const bool any = lh > 0.f;
      const float inv = any ? 1.f / lh : 0.f;
      float *dst = p.out + (size_t)orow[half] * D + 2 * c4;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd)
        *reinterpret_cast<float2 *>(dst + nd * 8) =
            make_float2(st.o[nd][2 * half] * inv, st.o[nd][2 * half + 1] * inv);
      if (p.lse && c4 == 0)
        p.lse[orow[half]] = any ? (st.m[half] + log2f(lh)) * 0.69314718055994530942f : -INFINITY;
    }
  };

  for (int k = 0;; ++k) {
    const int slot = k % S;
    mq::cp_async_wait<S - 2>();
    __syncthreads();  // unit k staged by every thread; unit k-1 finished by every warp
    const int ns = (slot + S - 1) % S;
    mq::issue_block<FMT, D>(p.k_pool, p.v_pool, p.row_bytes, bs, ahead.kvh, ahead_phys, ring, ns);
    if (threadIdx.x == 0) phys_ring[ns] = ahead_phys;
    if (ahead.tile >= 0) ahead.next(p, ts, n_tiles);
    ahead_phys = unit_phys(p, ahead);

    if (k > 0) cur.next(p, ts, n_tiles);
    if (cur.tile < 0) break;
    if (cur.b == 0) {
      if (k > 0) flush();
      // new tile: this warp's rows are (query, head) = (R / GP, R % GP)
      const float *qrow[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int R = 16 * warp + gid + 8 * half;
        const int j = cur.qt * TQ + R / GP;
        const int hg = R % GP;
        const int pos = cur.c - cur.n + j;
        const int i = p.q_start[cur.s] + j;
        const bool row_in = j < cur.n && hg < p.G && i >= 0 && i < p.n_tok;
        if (j < cur.n && hg < p.G && !row_in) report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
        const bool ok = row_in && pos >= 0;
        int lo = 0, hi = ok ? min(pos + 1, cur.c) : 0;
        if (ok && p.spans) {
          lo = max(p.spans[2 * i], 0);
          hi = min(hi, p.spans[2 * i + 1]);
        }
        if (ok && use_map) {
          // the runs of this row, clipped to [0, hi); bounds = their span
          int rl = INT_MAX, rh = INT_MIN;
          for (int r = 0; r < R_RUNS; ++r) {
            const int a = max(p.kv_map[((size_t)i * R_RUNS + r) * 2], 0);
            const int e = min(p.kv_map[((size_t)i * R_RUNS + r) * 2] +
                                  p.kv_map[((size_t)i * R_RUNS + r) * 2 + 1],
                              hi);
            if (c4 == 0) runs_s[R][r] = make_int2(a, e);
            if (e > a) {
              rl = min(rl, a);
              rh = max(rh, e);
            }
          }
          lo = rl;
          hi = rh;
        } else if (use_map && c4 == 0) {
          for (int r = 0; r < R_RUNS; ++r) runs_s[R][r] = make_int2(0, 0);
        }
        if (!(hi > lo)) lo = hi = 0;
        lo_r[half] = lo;
        hi_r[half] = hi;
        orow[half] = row_in ? i * p.Hq + cur.kvh * p.G + hg : -1;
        qrow[half] = ok ? p.q + ((size_t)i * p.Hq + (size_t)cur.kvh * p.G + hg) * D : nullptr;
      }
      mq::load_q<D>(st, qrow[0], qrow[1], p.qscale, c4);
      int wl = INT_MAX, wh = INT_MIN;
#pragma unroll
      for (int half = 0; half < 2; ++half)
        if (lo_r[half] < hi_r[half]) {
          wl = min(wl, lo_r[half]);
          wh = max(wh, hi_r[half]);
        }
#pragma unroll
      for (int o2 = 16; o2; o2 >>= 1) {
        wl = min(wl, __shfl_xor_sync(kAll, wl, o2));
        wh = max(wh, __shfl_xor_sync(kAll, wh, o2));
      }
      if (lane == 0) {
        win_s[2 * warp] = wl;
        win_s[2 * warp + 1] = wh;
      }
      __syncthreads();  // also publishes runs_s
      ulo = INT_MAX;
      uhi = INT_MIN;
#pragma unroll
      for (int w2 = 0; w2 < mq::kWarps; ++w2) {
        ulo = min(ulo, win_s[2 * w2]);
        uhi = max(uhi, win_s[2 * w2 + 1]);
      }
    }

    if (phys_ring[slot] < 0) continue;  // hole, flagged id or an empty tile's unit
    const int pos0 = cur.b * bs;
    uint32_t mk[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      if (use_map) {
        const int R = 16 * warp + gid + 8 * half;
        uint32_t m = 0u;
#pragma unroll
        for (int r = 0; r < R_RUNS; ++r) {
          const int2 ab = runs_s[R][r];
          m |= mq::range_mask(ab.x, ab.y, pos0, bs);
        }
        mk[half] = m;
      } else {
        mk[half] = mq::range_mask(lo_r[half], hi_r[half], pos0, bs);
      }
    }
    const bool any = __any_sync(kAll, (mk[0] | mk[1]) != 0u);

    uint8_t *raw = ring + (size_t)slot * C::RAW_STAGE;
    if constexpr (FMT != MT_KV_F16) {
      mq::convert_unit<FMT, D>(raw, tiles, scales, bs, pos0, ulo, uhi);
      __syncthreads();
    } else if (pos0 < ulo || pos0 + bs > uhi) {
      mq::zero_v_rows_f16<D>(raw, bs, pos0, ulo, uhi);
      __syncthreads();
    }
    if (!any) continue;
    const uint8_t *kt = FMT == MT_KV_F16 ? raw : tiles;
    const uint8_t *vt = FMT == MT_KV_F16 ? raw + mq::kMaxBs * C::RP
                        : FMT == MT_KV_Q8_0 ? tiles + mq::kMaxBs * C::TP
                                            : tiles + 2 * mq::kMaxBs * C::TP;
    mq::unit<FMT, D>(st, kt, vt, scales, bs, mk[0], mk[1], lane);
  }
  flush();
  mq::cp_async_wait<0>();
}

template <int FMT, int D, int GP>
mt_status launch_t(const PrefillParams &p, int n_ctas, cudaStream_t s) {
  auto kern = prefill_kernel<FMT, D, GP>;
  constexpr int smem = mq::Cfg<FMT, D>::SMEM;
  mt_status st = kernel_smem(reinterpret_cast<const void *>(kern), smem,
                             "cudaFuncSetAttribute(prefill smem)");
  if (st != MT_OK) return st;
  return cuda_check(launch_pdl(kern, dim3(n_ctas), dim3(mq::kThreads), smem, s, p),
                    "prefill kernel launch");
}

template <int FMT, int D>
mt_status launch_d(int gp, const PrefillParams &p, int n_ctas, cudaStream_t s) {
  switch (gp) {
    case 1: return launch_t<FMT, D, 1>(p, n_ctas, s);
    case 2: return launch_t<FMT, D, 2>(p, n_ctas, s);
    case 4: return launch_t<FMT, D, 4>(p, n_ctas, s);
    default: return launch_t<FMT, D, 8>(p, n_ctas, s);
  }
}

int pad_g(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 0; }

}  // namespace
}  // namespace mtkv

using namespace mtkv;

extern "C" size_t mt_paged_prefill_workspace_bytes(const mt_paged_prefill_args *a) {
  if (!a) return 0;
  const int G = a->n_kv_heads > 0 && a->n_heads % a->n_kv_heads == 0 ? a->n_heads / a->n_kv_heads : 0;
  return kPrefillWsBytes + prefill_rec_bytes(a, G > 0 ? pad_g(G) : 0) + tc_stage_bytes(a);
}

extern "C" mt_status mt_paged_attn_prefill(const mt_paged_prefill_args *a, void *workspace,
                                           size_t workspace_bytes, mt_stream stream) {
  if (!a) return fail(MT_ERR_INVALID_ARG, "prefill: null args");
  const size_t rb = mt_kv_row_bytes(a->fmt, a->n_kv_heads, a->head_dim);
  if (rb == 0) return fail(MT_ERR_INVALID_ARG, "prefill: unknown format or bad head shape");
  if (a->n_seqs < 0 || a->n_tokens < 0 || a->n_heads <= 0 || a->max_blocks < 0 ||
      a->n_phys_blocks < 0 || a->block_size <= 0)
    return fail(MT_ERR_INVALID_ARG, "prefill: negative or zero size");
  if (a->n_heads % a->n_kv_heads)
    return fail(MT_ERR_INVALID_ARG, "prefill: n_heads must be a multiple of n_kv_heads");
  const int G = a->n_heads / a->n_kv_heads;
  const int GP = pad_g(G);
  const bool d_ok = a->head_dim == 64 || a->head_dim == 128 ||
                    (a->head_dim == 256 && a->fmt != MT_KV_F32);
  if (!d_ok || (a->block_size != 16 && a->block_size != 32) || GP == 0)
    return fail(MT_ERR_UNSUPPORTED,
                "prefill: head_dim 64 or 128 (256 for f16 and q8_0 pools), block_size 16 or 32, "
                "at most 8 query heads per KV head");
  if (a->spans && a->kv_map)
    return fail(MT_ERR_INVALID_ARG, "prefill: spans and kv_map are two window modes: pass one");
  if ((long long)a->max_blocks * a->block_size > 0x7fffffffLL)
    return fail(MT_ERR_UNSUPPORTED, "prefill: max_blocks * block_size overflows int32");
  if (a->n_seqs == 0 || a->n_tokens == 0) return ok();
  if (!a->q || !a->k_pool || !a->v_pool || !a->block_table || !a->context_lens || !a->q_start ||
      !a->out)
    return fail(MT_ERR_INVALID_ARG, "prefill: null pointer");
  const size_t rec_bytes = prefill_rec_bytes(a, GP);
  const size_t stage_bytes = tc_stage_bytes(a);
  const size_t need = kPrefillWsBytes + rec_bytes + stage_bytes;
  if (!workspace || workspace_bytes < need)
    return fail(MT_ERR_INVALID_ARG, "prefill: workspace missing or too small (need " +
                                        std::to_string(need) + " bytes)");
  if (!aligned16(a->k_pool) || !aligned16(a->v_pool) || !aligned16(a->q) || !aligned16(a->out) ||
      !aligned16(workspace))
    return fail(MT_ERR_INVALID_ARG, "prefill: q, pools, out and workspace must be 16-byte aligned");
  DeviceInfo di;
  mt_status st = device_info(&di);
  if (st != MT_OK) return st;
  PrefillParams p;
  p.q = a->q;
  p.k_pool = static_cast<const uint8_t *>(a->k_pool);
  p.v_pool = static_cast<const uint8_t *>(a->v_pool);
  p.spans = a->spans;
  p.kv_map = a->kv_map;
  p.out = a->out;
  p.lse = a->lse;
  p.status = static_cast<uint32_t *>(workspace);
  p.n_tok = a->n_tokens;
  p.Hq = a->n_heads;
  p.Hkv = a->n_kv_heads;
  p.G = G;
  p.bs = a->block_size;
  p.max_blocks = a->max_blocks;
  p.n_phys = a->n_phys_blocks;
  p.row_bytes = (int)rb;
  p.qscale = a->scale * 1.4426950408889634f;
  p.rec = nullptr;
  p.rec_hdr = nullptr;
  p.rec_units = 0;
  if (rec_bytes && di.n_sm <= kSplitCtas) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.rec = reinterpret_cast<float *>(ws + kPrefillWsBytes);
    p.rec_hdr = reinterpret_cast<int *>(ws + 64);
    p.rec_units = 2 * kSplitCtas;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // f16 pools, and q8_0 / f32 pools staged as f16 / high-low f16 rows, run
  // the tcgen05 kernel
  const bool tc = a->fmt == MT_KV_F16 ? prefill_tc_supported(a->fmt, a->head_dim, a->block_size)
                                      : stage_bytes > 0;
  const bool pair = a->fmt == MT_KV_F32;
  if (!tc && a->head_dim != 256)
    return fail(MT_ERR_UNSUPPORTED,
                "prefill: q8_0 / f32 call too large to stage (n_seqs * max_blocks * block_size "
                "cells must stay below 2^31)");
  const int32_t *table = a->block_table;
  if (stage_bytes) {
    uint8_t *ws = static_cast<uint8_t *>(workspace) + kPrefillWsBytes + rec_bytes;
    const size_t tb = ((size_t)a->n_seqs * a->max_blocks * 4 + 255) & ~(size_t)255;
    const size_t pb = (stage_bytes - tb) / 2;
    int32_t *table16 = reinterpret_cast<int32_t *>(ws);
    uint8_t *k16 = ws + tb, *v16 = ws + tb + pb;
    if (pair)
      st = launch_stage_f32_pair(static_cast<const float *>(a->k_pool),
                                 static_cast<const float *>(a->v_pool), a->block_table,
                                 a->context_lens, a->n_seqs, a->max_blocks, a->block_size,
                                 a->n_phys_blocks, a->n_kv_heads, a->head_dim, k16, v16, table16,
                                 p.status, di.n_sm * 8, s);
    else
      st = launch_stage_q8_f16(p.k_pool, p.v_pool, a->block_table, a->context_lens, a->n_seqs,
                               a->max_blocks, a->block_size, a->n_phys_blocks, a->n_kv_heads,
                               a->head_dim, (int)rb, k16, v16, table16, p.status, di.n_sm * 8, s);
    if (st != MT_OK) return st;
    table = table16;
    p.k_pool = k16;
    p.v_pool = v16;
    p.n_phys = (long long)a->n_seqs * a->max_blocks;
    p.row_bytes = a->n_kv_heads * a->head_dim * (pair ? 4 : 2);
  }
  // sequences are independent: launch in chunks of kMaxPrefillSeqs (query
  // rows stay absolute, so only the per-sequence arrays are offset)
  for (int s0 = 0; s0 < a->n_seqs; s0 += kMaxPrefillSeqs) {
    p.B = std::min(kMaxPrefillSeqs, a->n_seqs - s0);
    p.table = table + (size_t)s0 * a->max_blocks;
    p.ctx = a->context_lens + s0;
    p.q_start = a->q_start + s0;
    if (tc) {
      // the tcgen05 kernel, one CTA (all 512 tensor-memory columns, ~198 KB
      // of shared memory for head_dim 128) per SM, then the merge of split
      // tiles (returns at once when nothing was split)
      st = launch_prefill_tc(p, a->head_dim, GP, pair, di.n_sm, s);
      if (st != MT_OK) return st;
      st = launch_prefill_tc_combine(p, a->head_dim, di.n_sm, s);
      if (st != MT_OK) return st;
      continue;
    }
    // head_dim 256 (f16, q8_0): the mma.sync kernel
    const int n_ctas = di.n_sm * 2;
    st = a->fmt == MT_KV_F16 ? launch_d<MT_KV_F16, 256>(GP, p, n_ctas, s)
                             : launch_d<MT_KV_Q8_0, 256>(GP, p, n_ctas, s);
    if (st != MT_OK) return st;
  }
  return ok();
}
