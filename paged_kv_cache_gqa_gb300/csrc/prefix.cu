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
#include "mma.cuh"
#include "prefix.h"

namespace mtkv {
namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kPWarps = kPrefixRows / 16;  // 4 consumer warps, 16 rows each
constexpr int kPThreads = 32 * kPWarps;
constexpr int kMaxBs = 32;
constexpr int kUnitChunk = 256;  // units whose block ids sit in shared memory at once

template <int FMT, int D>
struct PCfg {
  static constexpr int NG = D / 32;                       // q8_0 groups per head
  static constexpr int HB = FMT == MT_KV_F32 ? 4 * D : FMT == MT_KV_F16 ? 2 * D : NG * 34;
  static constexpr int TP = 2 * D + 16;                   // f16 tile pitch (bytes)
  // staged raw row pitch: f16 rows are staged straight into the tile layout
  static constexpr int RP = FMT == MT_KV_F16 ? TP : HB;
  // cp.async granule: head slices of q8_0 rows are 8-byte aligned when
  // d = 128 (136-byte slices) and 4-byte aligned when d = 64 (68 bytes)
  static constexpr int CH = FMT == MT_KV_Q8_0 ? (HB % 8 == 0 ? 8 : 4) : 16;
  static constexpr int RAW_STAGE = 2 * kMaxBs * RP;       // K and V
  // ring depth: about 64 KB of staged blocks (f32 blocks are 32 KB)
  static constexpr int STAGES = FMT == MT_KV_F32 ? 3 : FMT == MT_KV_F16 ? 4 : 6;
  static constexpr int N_TILES = FMT == MT_KV_F32 ? 4 : FMT == MT_KV_Q8_0 ? 2 : 0;
  static constexpr int TILE_BYTES = N_TILES * kMaxBs * TP;
  static constexpr int SCALE_BYTES = FMT == MT_KV_Q8_0 ? 2 * NG * kMaxBs * 4 : 0;
  static constexpr int SMEM = STAGES * RAW_STAGE + TILE_BYTES + SCALE_BYTES;
};

template <int CH>
__device__ __forceinline__ void cp_async(uint32_t dst, const void *src) {
  if constexpr (CH == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(CH)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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

// Issue the copies of unit u's K and V head slices (block `phys`, -1: none)
// into ring slot `slot`; one commit group per call, empty for holes and
// units past the range.
template <int FMT, int D>
__device__ __forceinline__ void issue_unit(const PrefixParams &p, int kvh, int phys,
                                           uint8_t *ring, int slot) {
  using C = PCfg<FMT, D>;
  if (phys >= 0) {
    constexpr int PER_ROW = C::HB / C::CH;
    const int n = p.bs * PER_ROW;
    const uint32_t base = smem_u32(ring + (size_t)slot * C::RAW_STAGE);
    const size_t cell0 = (size_t)phys * p.bs;
    for (int i = threadIdx.x; i < n; i += kPThreads) {
      const int r = i / PER_ROW, off = (i % PER_ROW) * C::CH;
      const size_t g = (cell0 + r) * (size_t)p.row_bytes + (size_t)kvh * C::HB + off;
      const uint32_t d = base + (uint32_t)(r * C::RP + off);
      cp_async<C::CH>(d, p.k_pool + g);
      cp_async<C::CH>(d + kMaxBs * C::RP, p.v_pool + g);
    }
  }
  cp_async_commit();
}

// q8_0: one (token, group) of a staged K or V slice -> 32 exact f16 codes in
// the tile row and the float32 scale. int8 -> f16 without the conversion
// unit: (q + 128) becomes the low byte of an f16 whose exponent gives 1024,
// so the half equals 1152 + q; subtracting 1152 is exact.
__device__ __forceinline__ void q8_convert_group(const uint8_t *raw, uint8_t *tile_row,
                                                 float *scale, int grp) {
  const uint8_t *blk = raw + grp * 34;
  // Read 9 aligned 32-bit words covering the block. A block that starts on a
  // word boundary holds its scale in the low half of word 0 and its codes
  // straddle word pairs (funnel shift); one that starts 2 bytes into a word
  // is read from 2 bytes earlier: scale in the high half of word 0, codes in
  // words 1..8.
  const bool odd = (reinterpret_cast<uintptr_t>(blk) & 3u) != 0;
  const uint32_t *w = reinterpret_cast<const uint32_t *>(blk - (odd ? 2 : 0));
  uint32_t x[9];
#pragma unroll
  for (int i = 0; i < 9; ++i) x[i] = w[i];
  uint32_t dbits, c[8];
  if (odd) {
    dbits = x[0] >> 16;  // blk starts in the high half of word 0
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = x[i + 1];
  } else {
    dbits = x[0] & 0xffffu;
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = __funnelshift_r(x[i], x[i + 1], 16);
  }
  *scale = __half2float(__ushort_as_half((unsigned short)dbits));
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  uint32_t out[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t v = c[i] ^ 0x80808080u;
    uint32_t lo = __byte_perm(v, 0x64646464u, 0x4140);
    uint32_t hi = __byte_perm(v, 0x64646464u, 0x4342);
    out[2 * i] = h2_bits(__hsub2(*reinterpret_cast<__half2 *>(&lo), bias));
    out[2 * i + 1] = h2_bits(__hsub2(*reinterpret_cast<__half2 *>(&hi), bias));
  }
  uint4 *dst = reinterpret_cast<uint4 *>(tile_row + grp * 64);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    dst[i] = make_uint4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
}

// Convert the staged unit in `raw` into the f16 tiles the MMAs read.
// V rows whose position lies outside [vlo, vhi) (no row of the tile reads
// them) are written as zeros, so that a zero probability never meets a
// non-finite value left in an unwritten cell.
template <int FMT, int D>
__device__ __forceinline__ void convert_unit(const uint8_t *raw, uint8_t *tiles, float *scales,
                                             int bs, int pos0, int vlo, int vhi) {
  using C = PCfg<FMT, D>;
  if constexpr (FMT == MT_KV_Q8_0) {
    // tiles: K codes, V codes; scales: [K|V][group][token]
    const int n = bs * C::NG;  // (token, group) items of K, then of V
    for (int i2 = threadIdx.x; i2 < 2 * n; i2 += kPThreads) {
      const int kv = i2 >= n;
      const int i = i2 - kv * n;
      const int r = i / C::NG;  // NG is a power of two
      const int grp = i % C::NG;
      float *sc = scales + (kv * C::NG + grp) * kMaxBs + r;
      q8_convert_group(raw + kv * kMaxBs * C::RP + r * C::RP,
                       tiles + kv * kMaxBs * C::TP + r * C::TP, sc, grp);
      // codes are always finite; a zero scale silences the row
      if (kv == 1 && (pos0 + r < vlo || pos0 + r >= vhi)) *sc = 0.f;
    }
  } else if constexpr (FMT == MT_KV_F32) {
    // tiles: K hi, K lo, V hi, V lo
    constexpr int Q4 = D / 4;
    const int n = bs * Q4;
    for (int i2 = threadIdx.x; i2 < 2 * n; i2 += kPThreads) {
      const int kv = i2 >= n;
      const int i = i2 - kv * n;
      const int r = i / Q4;
      const int e = (i % Q4) * 4;
      const float4 x =
          *reinterpret_cast<const float4 *>(raw + kv * kMaxBs * C::RP + r * C::RP + e * 4);
      uint32_t h0, l0, h1, l1;
      split_h2(x.x, x.y, h0, l0);
      split_h2(x.z, x.w, h1, l1);
      if (kv == 1 && (pos0 + r < vlo || pos0 + r >= vhi)) h0 = l0 = h1 = l1 = 0u;
      uint8_t *hi = tiles + (2 * kv) * kMaxBs * C::TP + r * C::TP + e * 2;
      uint8_t *lo = tiles + (2 * kv + 1) * kMaxBs * C::TP + r * C::TP + e * 2;
      *reinterpret_cast<uint2 *>(hi) = make_uint2(h0, h1);
      *reinterpret_cast<uint2 *>(lo) = make_uint2(l0, l1);
    }
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
__global__ void __launch_bounds__(kPThreads, 2) prefix_kernel(const __grid_constant__ PrefixParams p) {
  using C = PCfg<FMT, D>;
  constexpr int KS = D / 16;  // k-steps over the head dims
  constexpr int ND = D / 8;   // 8-dim output tiles
  constexpr int TQ = kPrefixRows / GP;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  uint8_t *tiles = smem + C::STAGES * C::RAW_STAGE;
  float *scales = reinterpret_cast<float *>(tiles + C::TILE_BYTES);
  pdl_enter();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, c4 = lane & 3;
  const long long u_beg = (long long)blockIdx.x * p.c.per;
  const long long u_end = min(p.c.n_units, u_beg + p.c.per);
  if (u_beg >= u_end) return;
  const int bs = p.bs;

  constexpr int S = C::STAGES;
  // block ids of units [chunk0, chunk0 + kUnitChunk + S), refilled as the
  // loop walks the range (the copies run S-1 units ahead)
  __shared__ int phys_s[kUnitChunk + S];
  long long chunk0 = u_beg;
  load_unit_blocks(p, chunk0, (int)min((long long)kUnitChunk + S, u_end - chunk0), u_end, phys_s);
  __syncthreads();
  auto phys_of = [&](long long u) { return u < u_end ? phys_s[u - chunk0] : -1; };
  UnitIter cur, ahead;  // the unit being computed, the next one to copy
  cur.init(p, u_beg);
  ahead = cur;
#pragma unroll
  for (int i = 0; i < S - 1; ++i) {
    issue_unit<FMT, D>(p, ahead.kvh, phys_of(u_beg + i), ring, i);
    if (u_beg + i + 1 < u_end) ahead.next(p);
  }

  uint32_t qh[KS][4], ql[KS][4];
  float o[ND][4];
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  int lo_r[2] = {0, 0}, hi_r[2] = {0, 0};
  int cur_T = -1;
  int rec_T = -1;  // tile of the segment being accumulated
  int ulo = 0, uhi = 0;  // union of the current tile's windows
  __shared__ int win_s[2 * kPWarps];

  // write this warp's rows of the current segment as one partial record
  auto flush = [&]() {
    float l0 = l_r[0], l1 = l_r[1];
    l0 += __shfl_xor_sync(kAll, l0, 1);
    l0 += __shfl_xor_sync(kAll, l0, 2);
    l1 += __shfl_xor_sync(kAll, l1, 1);
    l1 += __shfl_xor_sync(kAll, l1, 2);
    const size_t slot = (size_t)blockIdx.x + rec_T;
    const int R0 = 16 * warp + gid, R1 = R0 + 8;
    if (c4 == 0) {
      *reinterpret_cast<float2 *>(p.c.rec_ml + (slot * kPrefixRows + R0) * 2) =
          make_float2(m_r[0], l0);
      *reinterpret_cast<float2 *>(p.c.rec_ml + (slot * kPrefixRows + R1) * 2) =
          make_float2(m_r[1], l1);
    }
    float *o0 = p.c.rec_o + (slot * kPrefixRows + R0) * D + 2 * c4;
    float *o1 = p.c.rec_o + (slot * kPrefixRows + R1) * D + 2 * c4;
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      *reinterpret_cast<float2 *>(o0 + nd * 8) = make_float2(o[nd][0], o[nd][1]);
      *reinterpret_cast<float2 *>(o1 + nd * 8) = make_float2(o[nd][2], o[nd][3]);
    }
  };

  for (long long u = u_beg; u < u_end; ++u) {
    const int slot = (int)((u - u_beg) % S);
    cp_async_wait<S - 2>();
    __syncthreads();  // unit u staged by every thread; unit u-1 finished by every warp
    if (u - chunk0 == kUnitChunk) {
      // the next chunk of block ids (units already issued are re-read: same values)
      chunk0 = u;
      load_unit_blocks(p, chunk0, (int)min((long long)kUnitChunk + S, u_end - chunk0), u_end,
                       phys_s);
      __syncthreads();
    }
    issue_unit<FMT, D>(p, ahead.kvh, phys_of(u + S - 1), ring, (slot + S - 1) % S);
    if (u + S < u_end) ahead.next(p);

    if (u > u_beg) cur.next(p);
    const int T = cur.T, grp = cur.grp, qt = cur.qt, kvh = cur.kvh, b = cur.b;
    if (T != cur_T) {
      if (cur_T >= 0) flush();
      cur_T = rec_T = T;
      // new tile: this warp's rows are (sequence, head) = (R / GP, R % GP)
      const PrefixGroup g = p.c.g[grp];
      const int limit = g.nblk * bs;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int R = 16 * warp + gid + 8 * half;
        const int s = g.s0 + qt * TQ + R / GP;
        const int hg = R % GP;
        const bool ok = s < g.s1 && hg < p.G;
        if (ok) {
          prefix_window(p, s, limit, lo_r[half], hi_r[half]);
        } else {
          lo_r[half] = hi_r[half] = 0;
        }
        m_r[half] = -INFINITY;
        l_r[half] = 0.f;
        const float *qrow = p.q + ((size_t)(ok ? s : 0) * p.Hq + (size_t)kvh * p.G + hg) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
          if (ok) {
            x0 = *reinterpret_cast<const float2 *>(qrow + 16 * ks + 2 * c4);
            x1 = *reinterpret_cast<const float2 *>(qrow + 16 * ks + 2 * c4 + 8);
          }
          // A fragment: regs 0/2 hold row gid (cols 2c, 2c+8), 1/3 row gid+8
          split_h2(x0.x * p.qscale, x0.y * p.qscale, qh[ks][half], ql[ks][half]);
          split_h2(x1.x * p.qscale, x1.y * p.qscale, qh[ks][half + 2], ql[ks][half + 2]);
        }
      }
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
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
      for (int w2 = 0; w2 < kPWarps; ++w2) {
        ulo = min(ulo, win_s[2 * w2]);
        uhi = max(uhi, win_s[2 * w2 + 1]);
      }
    }

    if (phys_s[u - chunk0] < 0) continue;  // hole (or flagged id)
    const int pos0 = b * bs;
    // rows of this warp with no position in the block skip the math
    const bool any = __any_sync(kAll, (lo_r[0] < pos0 + bs && hi_r[0] > pos0) ||
                                          (lo_r[1] < pos0 + bs && hi_r[1] > pos0));

    uint8_t *raw = ring + (size_t)slot * C::RAW_STAGE;
    if constexpr (FMT != MT_KV_F16) {
      convert_unit<FMT, D>(raw, tiles, scales, bs, pos0, ulo, uhi);
      __syncthreads();
    } else if (pos0 < ulo || pos0 + bs > uhi) {
      // a block at the edge of the tile's windows: zero the V rows no row reads
      constexpr int U = C::HB / 16;
      for (int i = threadIdx.x; i < bs * U; i += kPThreads) {
        const int r = i / U;
        if (pos0 + r < ulo || pos0 + r >= uhi)
          *reinterpret_cast<uint4 *>(raw + (kMaxBs + r) * C::RP + (i % U) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
    }
    if (!any) continue;
    const uint8_t *kt = FMT == MT_KV_F16 ? raw : tiles;
    const uint8_t *vt = FMT == MT_KV_F16 ? raw + kMaxBs * C::RP
                        : FMT == MT_KV_Q8_0 ? tiles + kMaxBs * C::TP
                                            : tiles + 2 * kMaxBs * C::TP;
    const int NT = bs / 8;

    // ---- S = Q.K^T (base-2 logits), 8 tokens per n-tile; per 32 dims the
    // B fragments of all n-tiles are fetched first, then the MMAs of the
    // n-tiles interleave (independent accumulators)
    float sc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    const uint32_t ka = smem_u32(kt + (lane & 7) * C::TP) + (lane >> 3) * 16;
#pragma unroll
    for (int k2 = 0; k2 < D / 32; ++k2) {
      uint32_t bf[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
        if (nt < NT) ldsm_x4(ka + nt * 8 * C::TP + k2 * 64, bf[nt][0], bf[nt][1], bf[nt][2], bf[nt][3]);
      if constexpr (FMT == MT_KV_F16) {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          if (nt < NT) {
            mma_f16(sc[nt], qh[2 * k2], bf[nt][0], bf[nt][1]);
            mma_f16(sc[nt], qh[2 * k2 + 1], bf[nt][2], bf[nt][3]);
          }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          if (nt < NT) {
            mma_f16(sc[nt], ql[2 * k2], bf[nt][0], bf[nt][1]);
            mma_f16(sc[nt], ql[2 * k2 + 1], bf[nt][2], bf[nt][3]);
          }
      } else if constexpr (FMT == MT_KV_Q8_0) {
        // one 32-dim group: its own accumulators, then times the scales
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
          if (nt < NT) {
            mma_f16(acc[nt], qh[2 * k2], bf[nt][0], bf[nt][1]);
            mma_f16(acc[nt], qh[2 * k2 + 1], bf[nt][2], bf[nt][3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          if (nt < NT) {
            mma_f16(acc[nt], ql[2 * k2], bf[nt][0], bf[nt][1]);
            mma_f16(acc[nt], ql[2 * k2 + 1], bf[nt][2], bf[nt][3]);
          }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          if (nt < NT) {
            const float2 d =
                *reinterpret_cast<const float2 *>(scales + k2 * kMaxBs + nt * 8 + 2 * c4);
            sc[nt][0] = fmaf(d.x, acc[nt][0], sc[nt][0]);
            sc[nt][1] = fmaf(d.y, acc[nt][1], sc[nt][1]);
            sc[nt][2] = fmaf(d.x, acc[nt][2], sc[nt][2]);
            sc[nt][3] = fmaf(d.y, acc[nt][3], sc[nt][3]);
          }
      } else {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          if (nt < NT) {
            uint32_t l0, l1, l2, l3;
            ldsm_x4(ka + nt * 8 * C::TP + k2 * 64 + kMaxBs * C::TP, l0, l1, l2, l3);
            mma_f16(sc[nt], qh[2 * k2], bf[nt][0], bf[nt][1]);
            mma_f16(sc[nt], qh[2 * k2 + 1], bf[nt][2], bf[nt][3]);
            mma_f16(sc[nt], ql[2 * k2], bf[nt][0], bf[nt][1]);
            mma_f16(sc[nt], ql[2 * k2 + 1], bf[nt][2], bf[nt][3]);
            mma_f16(sc[nt], qh[2 * k2], l0, l1);
            mma_f16(sc[nt], qh[2 * k2 + 1], l2, l3);
          }
      }
    }

    // ---- mask, online softmax (rows gid and gid+8 of this warp)
    float mloc[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      if (nt >= NT) continue;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int half = e >> 1;
        const int pos = pos0 + nt * 8 + 2 * c4 + (e & 1);
        const bool v = pos >= lo_r[half] && pos < hi_r[half];
        sc[nt][e] = v ? sc[nt][e] : -INFINITY;
        mloc[half] = fmaxf(mloc[half], sc[nt][e]);
      }
    }
    float alpha[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float m = mloc[half];
      m = fmaxf(m, __shfl_xor_sync(kAll, m, 1));
      m = fmaxf(m, __shfl_xor_sync(kAll, m, 2));
      const float m_new = fmaxf(m_r[half], m);
      const bool none = m_new == -INFINITY;
      alpha[half] = none ? 1.f : exp2f(m_r[half] - m_new);
      m_r[half] = m_new;
      float lsum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        if (nt >= NT) continue;
        const float a = none ? 0.f : exp2f(sc[nt][2 * half] - m_new);
        const float bb = none ? 0.f : exp2f(sc[nt][2 * half + 1] - m_new);
        sc[nt][2 * half] = a;
        sc[nt][2 * half + 1] = bb;
        lsum += a + bb;
      }
      l_r[half] = l_r[half] * alpha[half] + lsum;
    }
    if (!__all_sync(kAll, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        o[nd][0] *= alpha[0];
        o[nd][1] *= alpha[0];
        o[nd][2] *= alpha[1];
        o[nd][3] *= alpha[1];
      }
    }

    // ---- O += P.V, 16 tokens per k-step; P from the score registers
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      if (2 * kk >= NT) continue;
      const float *pa = sc[2 * kk], *pb = sc[2 * kk + 1];
      const uint32_t va = smem_u32(vt + (16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8) * C::TP) +
                          (lane >> 4) * 16;
      if constexpr (FMT == MT_KV_F16) {
        uint32_t a[4];
        a[0] = h2_bits(__floats2half2_rn(pa[0], pa[1]));
        a[1] = h2_bits(__floats2half2_rn(pa[2], pa[3]));
        a[2] = h2_bits(__floats2half2_rn(pb[0], pb[1]));
        a[3] = h2_bits(__floats2half2_rn(pb[2], pb[3]));
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(va + dn * 32, b0, b1, b2, b3);
          mma_f16(o[2 * dn], a, b0, b1);
          mma_f16(o[2 * dn + 1], a, b2, b3);
        }
      } else if constexpr (FMT == MT_KV_Q8_0) {
        const float *vsc = scales + C::NG * kMaxBs;
#pragma unroll
        for (int grp = 0; grp < C::NG; ++grp) {
          const float2 da = *reinterpret_cast<const float2 *>(vsc + grp * kMaxBs + 16 * kk + 2 * c4);
          const float2 db =
              *reinterpret_cast<const float2 *>(vsc + grp * kMaxBs + 16 * kk + 8 + 2 * c4);
          uint32_t a[4];
          a[0] = h2_bits(__floats2half2_rn(pa[0] * da.x, pa[1] * da.y));
          a[1] = h2_bits(__floats2half2_rn(pa[2] * da.x, pa[3] * da.y));
          a[2] = h2_bits(__floats2half2_rn(pb[0] * db.x, pb[1] * db.y));
          a[3] = h2_bits(__floats2half2_rn(pb[2] * db.x, pb[3] * db.y));
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int dn = 2 * grp + j;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(va + dn * 32, b0, b1, b2, b3);
            mma_f16(o[2 * dn], a, b0, b1);
            mma_f16(o[2 * dn + 1], a, b2, b3);
          }
        }
      } else {
        uint32_t ah[4], al[4];
        split_h2(pa[0], pa[1], ah[0], al[0]);
        split_h2(pa[2], pa[3], ah[1], al[1]);
        split_h2(pb[0], pb[1], ah[2], al[2]);
        split_h2(pb[2], pb[3], ah[3], al[3]);
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
          ldsm_x4_t(va + dn * 32, b0, b1, b2, b3);
          ldsm_x4_t(va + dn * 32 + kMaxBs * C::TP, c0, c1, c2, c3);
          mma_f16(o[2 * dn], ah, b0, b1);
          mma_f16(o[2 * dn], al, b0, b1);
          mma_f16(o[2 * dn], ah, c0, c1);
          mma_f16(o[2 * dn + 1], ah, b2, b3);
          mma_f16(o[2 * dn + 1], al, b2, b3);
          mma_f16(o[2 * dn + 1], ah, c2, c3);
        }
      }
    }
  }
  if (cur_T >= 0) flush();
  cp_async_wait<0>();
}

}  // namespace

bool prefix_supported(int head_dim, int block_size, int gp) {
  return (head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32) &&
         (gp == 1 || gp == 2 || gp == 4 || gp == 8);
}

int prefix_smem_bytes(mt_kv_format fmt, int head_dim) {
  const bool d64 = head_dim == 64;
  switch (fmt) {
    case MT_KV_F32: return d64 ? PCfg<MT_KV_F32, 64>::SMEM : PCfg<MT_KV_F32, 128>::SMEM;
    case MT_KV_F16: return d64 ? PCfg<MT_KV_F16, 64>::SMEM : PCfg<MT_KV_F16, 128>::SMEM;
    default: return d64 ? PCfg<MT_KV_Q8_0, 64>::SMEM : PCfg<MT_KV_Q8_0, 128>::SMEM;
  }
}

int prefix_ctas_per_sm() { return 2; }

namespace {

template <int FMT, int D, int GP>
mt_status launch_t(const PrefixParams &p, int n_ctas, cudaStream_t s) {
  static int configured_dev = -1;
  auto kern = prefix_kernel<FMT, D, GP>;
  constexpr int smem = PCfg<FMT, D>::SMEM;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    mt_status st =
        cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                   "cudaFuncSetAttribute(prefix smem)");
    if (st != MT_OK) return st;
    configured_dev = dev;
  }
  return cuda_check(launch_pdl(kern, dim3(n_ctas), dim3(kPThreads), smem, s, p),
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
  return head_dim == 64 ? launch_d<FMT, 64>(gp, p, n_ctas, s) : launch_d<FMT, 128>(gp, p, n_ctas, s);
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
