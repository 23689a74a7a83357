// Multi-query paged attention core, for sm_103a: staging of one KV head's
// slice of a block, its conversion to f16 tensor-core tiles, and the
// per-warp math of 16 query rows against one staged block. Shared by the
// shared-prefix (cascade) kernel and the multi-query (prefill) kernel.
//
// What one call of mq::unit computes — for 16 rows (query token, head) of a
// warp and the tokens of one block that each row may read (a 32-bit mask per
// row), the online-softmax update of "Tiered KV cache — architecture",
// section "The paged-attention block model" / "Kernel dispatch" (masked
// positions have logit -infinity): S = scale * q . k in base 2, running max
// m and sum l, O = O * 2^(m_old - m_new) + sum_t 2^(S_t - m_new) v_t.
//
// Layout and numerics (GB300): mma.sync.m16n8k16 with f16 operands and f32
// accumulation; Q enters as a high/low f16 pair (q = hi + lo to ~2^-22) so
// scores keep float32 accuracy; K and V tiles sit in shared memory with a
// row pitch of 2d+16 bytes (an odd number of 16-byte units: every ldmatrix
// phase is conflict-free). q8_0 tiles hold exact f16 codes with float32
// scales per (token, 32-dim group): the scale multiplies each group's partial
// score and, for P.V, the probability operand. f32 pools (1e-4) use high/low
// tile pairs and three products (hi.hi + lo.hi + hi.lo).
#pragma once

#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "mma.cuh"

namespace mtkv {
namespace mq {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kWarps = 4;         // 16 rows each
constexpr int kThreads = 32 * kWarps;
constexpr int kRows = 16 * kWarps;
constexpr int kMaxBs = 32;

template <int FMT, int D>
struct Cfg {
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
  // head_dim above 128: the Q fragments would not fit in registers beside O,
  // so each warp keeps its 16 rows of Q (high rows, then low rows, pitch
  // 2d+16 bytes) in shared memory and reads them with ldmatrix per k-step
  static constexpr bool QS = D > 128;
  static constexpr int QTP = 2 * D + 16;
  static constexpr int QS_WARP = 2 * 16 * QTP;
  static constexpr int QS_BYTES = QS ? kWarps * QS_WARP : 0;
  static constexpr int SMEM = STAGES * RAW_STAGE + TILE_BYTES + SCALE_BYTES + QS_BYTES;
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


// Copy the K and V slices of KV head `kvh` of block `phys` (rows of
// `row_bytes`, `bs` per block) into ring slot `slot`; one commit group per
// call, empty when phys < 0.
template <int FMT, int D>
__device__ __forceinline__ void issue_block(const uint8_t *k_pool, const uint8_t *v_pool,
                                            int row_bytes, int bs, int kvh, int phys,
                                            uint8_t *ring, int slot) {
  using C = Cfg<FMT, D>;
  if (phys >= 0) {
    constexpr int PER_ROW = C::HB / C::CH;
    const int n = bs * PER_ROW;
    const uint32_t base = smem_u32(ring + (size_t)slot * C::RAW_STAGE);
    const size_t cell0 = (size_t)phys * bs;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const int r = i / PER_ROW, off = (i % PER_ROW) * C::CH;
      const size_t g = (cell0 + r) * (size_t)row_bytes + (size_t)kvh * C::HB + off;
      const uint32_t d = base + (uint32_t)(r * C::RP + off);
      cp_async<C::CH>(d, k_pool + g);
      cp_async<C::CH>(d + kMaxBs * C::RP, v_pool + g);
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
  using C = Cfg<FMT, D>;
  if constexpr (FMT == MT_KV_Q8_0) {
    // tiles: K codes, V codes; scales: [K|V][group][token]
    const int n = bs * C::NG;  // (token, group) items of K, then of V
    for (int i2 = threadIdx.x; i2 < 2 * n; i2 += kThreads) {
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
    for (int i2 = threadIdx.x; i2 < 2 * n; i2 += kThreads) {
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


// f16 pools stage straight into the tiles: zero the V rows of the unit whose
// position lies outside [vlo, vhi) (the caller then synchronises the CTA).
template <int D>
__device__ __forceinline__ void zero_v_rows_f16(uint8_t *raw, int bs, int pos0, int vlo,
                                                int vhi) {
  using C = Cfg<MT_KV_F16, D>;
  constexpr int U = C::HB / 16;
  for (int i = threadIdx.x; i < bs * U; i += kThreads) {
    const int r = i / U;
    if (pos0 + r < vlo || pos0 + r >= vhi)
      *reinterpret_cast<uint4 *>(raw + (kMaxBs + r) * C::RP + (i % U) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
  }
}

// Tokens [lo - pos0, hi - pos0) of a block starting at position pos0, as a
// bit mask over its bs <= 32 slots.
__device__ __forceinline__ uint32_t range_mask(int lo, int hi, int pos0, int bs) {
  const int a = max(lo - pos0, 0), b = min(hi - pos0, bs);
  if (b <= a) return 0u;
  const uint32_t upto = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
  return upto & ~((1u << a) - 1u);
}

// Per-thread state of a warp's 16 rows: this thread holds rows gid and
// gid + 8 (gid = lane / 4) of the MMA fragments.
template <int D>
struct Rows {
  static constexpr bool QS = D > 128;       // Q in shared memory (see Cfg::QS)
  static constexpr int QTP = 2 * D + 16;
  uint32_t qh[QS ? 1 : D / 16][4], ql[QS ? 1 : D / 16][4];  // A fragments of q*scale*log2(e)
  uint32_t qs;                            // QS: shared address of the warp's Q rows
  float o[D / 8][4];                      // unnormalised output
  float m[2], l[2];                       // running max (base 2), partial sums
};

// The A fragments (high and low) of k-step ks of this warp's Q.
template <int D>
__device__ __forceinline__ void q_frags(const Rows<D> &st, int ks, int lane, uint32_t (&h)[4],
                                        uint32_t (&l)[4]) {
  if constexpr (Rows<D>::QS) {
    // ldmatrix.x4: lanes 0-7 rows 0-7 / cols 0-7, 8-15 rows 8-15 / cols 0-7,
    // 16-23 rows 0-7 / cols 8-15, 24-31 rows 8-15 / cols 8-15
    const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t a = st.qs + (uint32_t)(r * Rows<D>::QTP + ks * 32 + (lane >> 4) * 16);
    ldsm_x4(a, h[0], h[1], h[2], h[3]);
    ldsm_x4(a + 16 * Rows<D>::QTP, l[0], l[1], l[2], l[3]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      h[i] = st.qh[ks][i];
      l[i] = st.ql[ks][i];
    }
  }
}

// Start rows gid / gid+8 with query rows q0 / q1 (null: padding row).
template <int D>
__device__ __forceinline__ void load_q(Rows<D> &st, const float *q0, const float *q1,
                                       float qscale, int c4) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const float *qrow = half ? q1 : q0;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
      if (qrow) {
        x0 = *reinterpret_cast<const float2 *>(qrow + 16 * ks + 2 * c4);
        x1 = *reinterpret_cast<const float2 *>(qrow + 16 * ks + 2 * c4 + 8);
      }
      if constexpr (Rows<D>::QS) {
        // rows gid / gid+8 of the warp's Q tile, cols 16ks + 2c and +8
        uint32_t h0, l0, h1, l1;
        split_h2(x0.x * qscale, x0.y * qscale, h0, l0);
        split_h2(x1.x * qscale, x1.y * qscale, h1, l1);
        const int r = (threadIdx.x & 31) / 4 + 8 * half;
        uint8_t *t = reinterpret_cast<uint8_t *>(__cvta_shared_to_generic(st.qs)) +
                     r * Rows<D>::QTP + (16 * ks + 2 * c4) * 2;
        *reinterpret_cast<uint32_t *>(t) = h0;
        *reinterpret_cast<uint32_t *>(t + 16) = h1;
        *reinterpret_cast<uint32_t *>(t + 16 * Rows<D>::QTP) = l0;
        *reinterpret_cast<uint32_t *>(t + 16 * Rows<D>::QTP + 16) = l1;
      } else {
        // A fragment: regs 0/2 hold row gid (cols 2c, 2c+8), 1/3 row gid+8
        split_h2(x0.x * qscale, x0.y * qscale, st.qh[ks][half], st.ql[ks][half]);
        split_h2(x1.x * qscale, x1.y * qscale, st.qh[ks][half + 2], st.ql[ks][half + 2]);
      }
    }
    st.m[half] = -INFINITY;
    st.l[half] = 0.f;
  }
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) st.o[nd][0] = st.o[nd][1] = st.o[nd][2] = st.o[nd][3] = 0.f;
  if constexpr (Rows<D>::QS) __syncwarp();  // the warp's Q rows are written
}

// Row sums of the quad (the 4 threads sharing rows gid, gid + 8).
template <int D>
__device__ __forceinline__ float2 row_sums(const Rows<D> &st) {
  float l0 = st.l[0], l1 = st.l[1];
  l0 += __shfl_xor_sync(kAll, l0, 1);
  l0 += __shfl_xor_sync(kAll, l0, 2);
  l1 += __shfl_xor_sync(kAll, l1, 1);
  l1 += __shfl_xor_sync(kAll, l1, 2);
  return make_float2(l0, l1);
}

// One staged block against this warp's rows. kt / vt: the K and V tiles (f32:
// the high tiles, the low ones kMaxBs rows further); scales: q8_0 scales
// [K|V][group][token]; mk0 / mk1: readable tokens of rows gid / gid + 8.
template <int FMT, int D>
__device__ __forceinline__ void unit(Rows<D> &st, const uint8_t *kt, const uint8_t *vt,
                                     const float *scales, int bs, uint32_t mk0, uint32_t mk1,
                                     int lane) {
  using C = Cfg<FMT, D>;
  constexpr int ND = D / 8;
  const int c4 = lane & 3;
  const int NT = bs / 8;
  auto &o = st.o;
  auto &m_r = st.m;
  auto &l_r = st.l;
  // ---- S = Q.K^T (base-2 logits), 8 tokens per n-tile; per 32 dims the
  // B fragments of all n-tiles are fetched first, then the MMAs of the
  // n-tiles interleave (independent accumulators)
  float sc[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
  const uint32_t ka = smem_u32(kt + (lane & 7) * C::TP) + (lane >> 3) * 16;
#pragma unroll
  for (int k2 = 0; k2 < D / 32; ++k2) {
    // Q's A fragments of the group's two k-steps (registers, or shared
    // memory for head_dim 256)
    uint32_t qh[2][4], ql[2][4];
    q_frags<D>(st, 2 * k2, lane, qh[0], ql[0]);
    q_frags<D>(st, 2 * k2 + 1, lane, qh[1], ql[1]);
    uint32_t bf[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
      if (nt < NT) ldsm_x4(ka + nt * 8 * C::TP + k2 * 64, bf[nt][0], bf[nt][1], bf[nt][2], bf[nt][3]);
    if constexpr (FMT == MT_KV_F16) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
        if (nt < NT) {
          mma_f16(sc[nt], qh[0], bf[nt][0], bf[nt][1]);
          mma_f16(sc[nt], qh[1], bf[nt][2], bf[nt][3]);
        }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
        if (nt < NT) {
          mma_f16(sc[nt], ql[0], bf[nt][0], bf[nt][1]);
          mma_f16(sc[nt], ql[1], bf[nt][2], bf[nt][3]);
        }
    } else if constexpr (FMT == MT_KV_Q8_0) {
      // one 32-dim group: its own accumulators, then times the scales
      float acc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        if (nt < NT) {
          mma_f16(acc[nt], qh[0], bf[nt][0], bf[nt][1]);
          mma_f16(acc[nt], qh[1], bf[nt][2], bf[nt][3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
        if (nt < NT) {
          mma_f16(acc[nt], ql[0], bf[nt][0], bf[nt][1]);
          mma_f16(acc[nt], ql[1], bf[nt][2], bf[nt][3]);
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
          mma_f16(sc[nt], qh[0], bf[nt][0], bf[nt][1]);
          mma_f16(sc[nt], qh[1], bf[nt][2], bf[nt][3]);
          mma_f16(sc[nt], ql[0], bf[nt][0], bf[nt][1]);
          mma_f16(sc[nt], ql[1], bf[nt][2], bf[nt][3]);
          mma_f16(sc[nt], qh[0], l0, l1);
          mma_f16(sc[nt], qh[1], l2, l3);
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
      const uint32_t mk = half ? mk1 : mk0;
      const bool v = (mk >> (nt * 8 + 2 * c4 + (e & 1))) & 1u;
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

}  // namespace mq
}  // namespace mtkv
