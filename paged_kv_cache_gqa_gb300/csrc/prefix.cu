// Prefix kernel of the shared-prefix (cascade) decode, for sm_103a.
//
// What is computed — for every sequence s of a group and query head h, the
// unnormalised attention partial (max m, sum l, output O = sum 2^(t-m) v)
// over the positions of the group's shared prefix that lie in s's window:
// "Tiered KV cache — architecture", section "The paged-attention block
// model" (block table, holes read as -infinity, point 2: refcounted shared
// blocks) and "KV Cache Design — cells, format, sessions", section 1 (the
// [lo, hi) window of each query). The combine merges these partials with the
// suffix decode's by log-sum-exp, so the cascade computes exactly what the
// plain decode computes.
//
// How (GB300): a tile is 64 (sequence, query head) rows of one KV head: the
// decode queries of up to 64/GP sequences that share the block. Four warps
// own 16 rows each and run S = Q.K^T and O += P.V on the tensor cores
// (mma.sync.m16n8k16, f16 operands, f32 accumulation):
//   * Q enters as a high/low f16 pair (q = hi + lo to ~2^-22), both
//     multiplied into every K tile, so scores keep float32 accuracy;
//   * f16 pools: K and V head slices are copied (cp.async, 16 B) straight
//     into row-padded tiles (pitch 2d+16 bytes: an odd number of 16-byte
//     units, so ldmatrix phases are conflict-free);
//   * q8_0 pools: the raw 34-byte blocks are copied, then converted once per
//     CTA into exact f16 codes plus float32 scales; the scale multiplies each
//     32-dim group's partial score (one accumulator per group) and, for P.V,
//     the probability operand of that group;
//   * f32 pools (1e-4): K and V become high/low f16 tile pairs and both
//     products use three MMAs (hi.hi + lo.hi + hi.lo).
// The block ring holds about 64 KB of staged blocks (6 q8_0, 4 f16, 3 f32
// stages); each CTA reads its units' block ids into shared memory once, so
// no global load sits between a stage's release and its next copy. Every
// block is fetched once per tile, i.e. once for all the sequences of the tile
// instead of once per sequence.
#include <limits.h>
#include <math.h>

#include <algorithm>
#include <string>

#include "cascade.h"
#include "common.cuh"
#include "internal.h"
#include "mq.cuh"
#include "prefix.h"

namespace mtkv {
namespace {

constexpr int kUnitChunk = 256;  // units whose block ids sit in shared memory at once

// Physical block of unit u (its tile's leading sequence's table entry), or
// -1 for a hole, an id out of range (flagged) or a unit past the end. Also
// checks the group's promise for the sequence of the tile at `lane_seq`
// (identical table entry), flagging a mismatch.
__device__ __forceinline__ int unit_block(const PrefixParams &p, long long u, int lane_seq) {
  int T, grp, qt, kvh, b;
  cascade_unit(p.c, p.Hkv, u, T, grp, qt, kvh, b);
  if (T < 0) return -1;
  const PrefixGroup g = p.c.g[grp];
  const int phys = p.table[(size_t)g.s0 * p.max_blocks + b];
  const int s = g.s0 + qt * p.c.tq + lane_seq;
  if (lane_seq > 0 && lane_seq < p.c.tq && s < g.s1 &&
      p.table[(size_t)s * p.max_blocks + b] != phys)
    report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
  if (phys == MT_INVALID_BLOCK_ID) return -1;
  if (phys < 0 || (long long)phys >= p.n_phys) {
    report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
    return -1;
  }
  return phys;
}

// Walks consecutive units without divisions: (tile, group, query tile, KV
// head, block) of the current unit.
struct UnitIter {
  int T, grp, qt, kvh, b;
  __device__ __forceinline__ void init(const PrefixParams &p, long long u) {
    cascade_unit(p.c, p.Hkv, u, T, grp, qt, kvh, b);
  }
  __device__ __forceinline__ void next(const PrefixParams &p) {
    if (++b < p.c.g[grp].nblk) return;
    b = 0;
    ++T;
    if (++kvh < p.Hkv) return;
    kvh = 0;
    if (++qt < cascade_qtiles(p.c, grp)) return;
    qt = 0;
    // groups without a prefix have no units, but their tiles count in T
    for (++grp; grp < p.c.n_groups && p.c.g[grp].nblk == 0; ++grp)
      T += cascade_qtiles(p.c, grp) * p.Hkv;
    if (grp >= p.c.n_groups) T = -1;
  }
};

// Block ids of units [u0, u0 + n) into phys_s (n <= kUnitChunk + STAGES),
// with the group checks spread over the CTA's threads.
__device__ __forceinline__ void load_unit_blocks(const PrefixParams &p, long long u0, int n,
                                                 long long u_end, int *phys_s) {
  const int tq = p.c.tq;
  for (int i = threadIdx.x; i < n * tq; i += blockDim.x) {
    const int k = i / tq, j = i % tq;
    const long long u = u0 + k;
    const int ph = u < u_end ? unit_block(p, u, j) : -1;
    if (j == 0) phys_s[k] = ph;
  }
}

// Window of sequence s clipped to the shared prefix [0, limit): the positions
// the prefix partial covers (lo == hi: none).
__device__ __forceinline__ void prefix_window(const PrefixParams &p, int s, int limit, int &lo,
                                              int &hi) {
  int c = p.ctx[s];
  const int cmax = p.max_blocks * p.bs;
  c = c < 0 ? 0 : (c > cmax ? cmax : c);  // out-of-range lengths are flagged by the decode
  lo = 0;
  hi = c;
  if (p.spans) {
    lo = max(p.spans[2 * s], 0);
    hi = min(p.spans[2 * s + 1], c);
  }
  hi = min(hi, limit);
  if (hi <= lo) lo = hi = 0;
}

template <int FMT, int D, int GP>
__global__ void __launch_bounds__(mq::kThreads, 2)
    prefix_kernel(const __grid_constant__ PrefixParams p) {
  using C = mq::Cfg<FMT, D>;
  using mq::kAll;
  constexpr int TQ = kPrefixRows / GP;
  constexpr int S = C::STAGES;
  static_assert(kPrefixRows == mq::kRows, "a prefix tile is one multi-query tile");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  uint8_t *tiles = smem + S * C::RAW_STAGE;
  float *scales = reinterpret_cast<float *>(tiles + C::TILE_BYTES);
  pdl_enter();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, c4 = lane & 3;
  const long long u_beg = (long long)blockIdx.x * p.c.per;
  const long long u_end = min(p.c.n_units, u_beg + p.c.per);
  if (u_beg >= u_end) return;
  const int bs = p.bs;

  // block ids of units [chunk0, chunk0 + kUnitChunk + S), refilled as the
  // loop walks the range (the copies run S-1 units ahead)
  __shared__ int phys_s[kUnitChunk + S];
  __shared__ int win_s[2 * mq::kWarps];
  // kv_map windows: the runs of the tile's rows, clipped to the prefix
  constexpr int R_RUNS = MT_KV_MAP_MAX_SPANS;
  __shared__ int2 runs_s[kPrefixRows][R_RUNS];
  const bool use_map = p.kv_map != nullptr;
  long long chunk0 = u_beg;
  load_unit_blocks(p, chunk0, (int)min((long long)kUnitChunk + S, u_end - chunk0), u_end, phys_s);
  __syncthreads();
  auto phys_of = [&](long long u) { return u < u_end ? phys_s[u - chunk0] : -1; };
  UnitIter cur, ahead;  // the unit being computed, the next one to copy
  cur.init(p, u_beg);
  ahead = cur;
#pragma unroll
  for (int i = 0; i < S - 1; ++i) {
    mq::issue_block<FMT, D>(p.k_pool, p.v_pool, p.row_bytes, bs, ahead.kvh, phys_of(u_beg + i),
                            ring, i);
    if (u_beg + i + 1 < u_end) ahead.next(p);
  }

  mq::Rows<D> st;
  if constexpr (C::QS) st.qs = smem_u32(smem + C::SMEM - C::QS_BYTES) + warp * C::QS_WARP;
  int lo_r[2] = {0, 0}, hi_r[2] = {0, 0};
  int cur_T = -1;
  int ulo = 0, uhi = 0;  // union of the current tile's windows

  // this warp's rows of the current segment as one partial record
  auto flush = [&]() {
    const float2 l = mq::row_sums(st);
    const size_t slot = (size_t)blockIdx.x + cur_T;
    const int R0 = 16 * warp + gid, R1 = R0 + 8;
    if (c4 == 0) {
      *reinterpret_cast<float2 *>(p.c.rec_ml + (slot * kPrefixRows + R0) * 2) =
          make_float2(st.m[0], l.x);
      *reinterpret_cast<float2 *>(p.c.rec_ml + (slot * kPrefixRows + R1) * 2) =
          make_float2(st.m[1], l.y);
    }
    float *o0 = p.c.rec_o + (slot * kPrefixRows + R0) * D + 2 * c4;
    float *o1 = p.c.rec_o + (slot * kPrefixRows + R1) * D + 2 * c4;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      *reinterpret_cast<float2 *>(o0 + nd * 8) = make_float2(st.o[nd][0], st.o[nd][1]);
      *reinterpret_cast<float2 *>(o1 + nd * 8) = make_float2(st.o[nd][2], st.o[nd][3]);
    }
  };

  for (long long u = u_beg; u < u_end; ++u) {
    const int slot = (int)((u - u_beg) % S);
    mq::cp_async_wait<S - 2>();
    __syncthreads();  // unit u staged by every thread; unit u-1 finished by every warp
    if (u - chunk0 == kUnitChunk) {
      // the next chunk of block ids (units already issued are re-read: same values)
      chunk0 = u;
      load_unit_blocks(p, chunk0, (int)min((long long)kUnitChunk + S, u_end - chunk0), u_end,
                       phys_s);
      __syncthreads();
    }
    mq::issue_block<FMT, D>(p.k_pool, p.v_pool, p.row_bytes, bs, ahead.kvh,
                            phys_of(u + S - 1), ring, (slot + S - 1) % S);
    if (u + S < u_end) ahead.next(p);

    if (u > u_beg) cur.next(p);
    if (cur.T != cur_T) {
      if (cur_T >= 0) flush();
      cur_T = cur.T;
      // new tile: this warp's rows are (sequence, head) = (R / GP, R % GP)
      const PrefixGroup g = p.c.g[cur.grp];
      const float *qrow[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int R = 16 * warp + gid + 8 * half;
        const int s = g.s0 + cur.qt * TQ + R / GP;
        const int hg = R % GP;
        const bool ok = s < g.s1 && hg < p.G;
        lo_r[half] = hi_r[half] = 0;
        if (ok) prefix_window(p, s, g.nblk * bs, lo_r[half], hi_r[half]);
        if (use_map) {
          // the row's runs inside [0, min(ctx, prefix)); bounds = their span
          int rl = INT_MAX, rh = INT_MIN;
          for (int r = 0; r < R_RUNS; ++r) {
            int a = 0, e = 0;
            if (ok) {
              const int32_t *rp = p.kv_map + ((size_t)s * R_RUNS + r) * 2;
              a = max(rp[0], 0);
              e = min(rp[0] + rp[1], hi_r[half]);
            }
            if (c4 == 0) runs_s[R][r] = make_int2(a, e);
            if (e > a) {
              rl = min(rl, a);
              rh = max(rh, e);
            }
          }
          lo_r[half] = rh > rl ? rl : 0;
          hi_r[half] = rh > rl ? rh : 0;
        }
        qrow[half] = ok ? p.q + ((size_t)s * p.Hq + (size_t)cur.kvh * p.G + hg) * D : nullptr;
      }
      mq::load_q<D>(st, qrow[0], qrow[1], p.qscale, c4);
      // union of the tile's windows (V rows outside it are zeroed)
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
      __syncthreads();
      ulo = INT_MAX;
      uhi = INT_MIN;
#pragma unroll
      for (int w2 = 0; w2 < mq::kWarps; ++w2) {
        ulo = min(ulo, win_s[2 * w2]);
        uhi = max(uhi, win_s[2 * w2 + 1]);
      }
    }

    if (phys_s[u - chunk0] < 0) continue;  // hole (or flagged id)
    const int pos0 = cur.b * bs;
    uint32_t mk0, mk1;
    if (use_map) {
      const int R0 = 16 * warp + gid;
      mk0 = mk1 = 0u;
#pragma unroll
      for (int r = 0; r < R_RUNS; ++r) {
        const int2 a0 = runs_s[R0][r], a1 = runs_s[R0 + 8][r];
        mk0 |= mq::range_mask(a0.x, a0.y, pos0, bs);
        mk1 |= mq::range_mask(a1.x, a1.y, pos0, bs);
      }
    } else {
      mk0 = mq::range_mask(lo_r[0], hi_r[0], pos0, bs);
      mk1 = mq::range_mask(lo_r[1], hi_r[1], pos0, bs);
    }
    // rows of this warp with no position in the block skip the math
    const bool any = __any_sync(kAll, (mk0 | mk1) != 0u);

    uint8_t *raw = ring + (size_t)slot * C::RAW_STAGE;
    if constexpr (FMT != MT_KV_F16) {
      mq::convert_unit<FMT, D>(raw, tiles, scales, bs, pos0, ulo, uhi);
      __syncthreads();
    } else if (pos0 < ulo || pos0 + bs > uhi) {
      // a block at the edge of the tile's windows: zero the V rows no row reads
      mq::zero_v_rows_f16<D>(raw, bs, pos0, ulo, uhi);
      __syncthreads();
    }
    if (!any) continue;
    const uint8_t *kt = FMT == MT_KV_F16 ? raw : tiles;
    const uint8_t *vt = FMT == MT_KV_F16 ? raw + mq::kMaxBs * C::RP
                        : FMT == MT_KV_Q8_0 ? tiles + mq::kMaxBs * C::TP
                                            : tiles + 2 * mq::kMaxBs * C::TP;
    mq::unit<FMT, D>(st, kt, vt, scales, bs, mk0, mk1, lane);
  }
  if (cur_T >= 0) flush();
  mq::cp_async_wait<0>();
}

}  // namespace

bool prefix_supported(mt_kv_format fmt, int head_dim, int block_size, int gp) {
  const bool d = head_dim == 64 || head_dim == 128 || (head_dim == 256 && fmt != MT_KV_F32);
  return d && (block_size == 16 || block_size == 32) && (gp == 1 || gp == 2 || gp == 4 || gp == 8);
}

int prefix_smem_bytes(mt_kv_format fmt, int head_dim) {
  switch (fmt) {
    case MT_KV_F32:
      return head_dim == 64 ? mq::Cfg<MT_KV_F32, 64>::SMEM : mq::Cfg<MT_KV_F32, 128>::SMEM;
    case MT_KV_F16:
      return head_dim == 64    ? mq::Cfg<MT_KV_F16, 64>::SMEM
             : head_dim == 128 ? mq::Cfg<MT_KV_F16, 128>::SMEM
                               : mq::Cfg<MT_KV_F16, 256>::SMEM;
    default:
      return head_dim == 64    ? mq::Cfg<MT_KV_Q8_0, 64>::SMEM
             : head_dim == 128 ? mq::Cfg<MT_KV_Q8_0, 128>::SMEM
                               : mq::Cfg<MT_KV_Q8_0, 256>::SMEM;
  }
}

// head_dim 256 keeps Q in shared memory (about 200 KB per CTA): one per SM
int prefix_ctas_per_sm(int head_dim) { return head_dim == 256 ? 1 : 2; }

namespace {

template <int FMT, int D, int GP>
mt_status launch_t(const PrefixParams &p, int n_ctas, cudaStream_t s) {
  auto kern = prefix_kernel<FMT, D, GP>;
  constexpr int smem = mq::Cfg<FMT, D>::SMEM;
  mt_status st = kernel_smem(reinterpret_cast<const void *>(kern), smem,
                             "cudaFuncSetAttribute(prefix smem)");
  if (st != MT_OK) return st;
  return cuda_check(launch_pdl(kern, dim3(n_ctas), dim3(mq::kThreads), smem, s, p),
                    "prefix kernel launch");
}

template <int FMT, int D>
mt_status launch_d(int gp, const PrefixParams &p, int n_ctas, cudaStream_t s) {
  switch (gp) {
    case 1: return launch_t<FMT, D, 1>(p, n_ctas, s);
    case 2: return launch_t<FMT, D, 2>(p, n_ctas, s);
    case 4: return launch_t<FMT, D, 4>(p, n_ctas, s);
    default: return launch_t<FMT, D, 8>(p, n_ctas, s);
  }
}

template <int FMT>
mt_status launch_f(int head_dim, int gp, const PrefixParams &p, int n_ctas, cudaStream_t s) {
  if (head_dim == 64) return launch_d<FMT, 64>(gp, p, n_ctas, s);
  if constexpr (FMT != MT_KV_F32) {
    if (head_dim == 256) return launch_d<FMT, 256>(gp, p, n_ctas, s);
  }
  return launch_d<FMT, 128>(gp, p, n_ctas, s);
}

}  // namespace

mt_status launch_prefix(mt_kv_format fmt, int head_dim, int gp, const PrefixParams &p, int n_ctas,
                        cudaStream_t stream) {
  switch (fmt) {
    case MT_KV_F32: return launch_f<MT_KV_F32>(head_dim, gp, p, n_ctas, stream);
    case MT_KV_F16: return launch_f<MT_KV_F16>(head_dim, gp, p, n_ctas, stream);
    default: return launch_f<MT_KV_Q8_0>(head_dim, gp, p, n_ctas, stream);
  }
}

}  // namespace mtkv
