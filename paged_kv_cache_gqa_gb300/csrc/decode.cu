// Paged grouped-query decode attention (split-K over a flattened block
// stream) and its combine step, for sm_103a.
//
// What is computed — "Tiered KV cache — architecture", sections "The
// paged-attention block model" (per-sequence logical -> physical block
// table; position p in cell table[p/bs]*bs + p%bs) and "Kernel dispatch"
// (block table + context lengths; kInvalidBlockId positions get logit
// -infinity, i.e. zero weight); "KV Cache Design — cells, format, sessions",
// section 1 (each query's window [lo, hi)) and section 3 (f32 / f16 / q8_0
// storage; q8_0 is read packed and dequantised in registers).
//
// How (GB300-first design, not the pages' kernels):
//  * Work is the stream of all sequences' (window-clipped) logical blocks,
//    cut into equal contiguous ranges, one per persistent CTA (one CTA per
//    SM; two when a CTA has at most three consumer warps, so every scheduler
//    still runs two). Every CTA derives its range from the context lengths
//    itself, so long and short sequences balance without a planning launch.
//    A CTA's range covers all KV heads of its blocks: the block's cells for
//    all heads are one contiguous span of the pool.
//  * Warp specialisation: one producer warp walks the range, reads block
//    ids (32 at a time), skips holes, and fills a shared-memory ring of up
//    to 8 stages guarded by mbarriers: one swizzled 3-D tensor copy per K
//    and per V block (f16, and f32 up to head_dim 128), else bulk copies of
//    the rows the window needs.
//  * Consumers: f16 and f32 (head_dim <= 128) pools on the tensor cores
//    (mma.sync, one warp per KV head; f32 values split into high / low f16
//    halves), q8_0 (head_dim <= 128) on the tensor cores from per-warp
//    converted tiles, the rest on the FP32 pipes: lanes own 16-dim (8 when
//    the group has more than 4 heads) slices of the head for one token; the
//    G group heads' partial dot products are reduced across the token's
//    lanes by recursive halving; online softmax in base 2 with the max
//    shared by the group; P.V with each lane owning head_dim/32 output dims
//    of every head.
//  * Each (CTA, sequence) segment writes an unnormalised partial (o, m, l);
//    the combine kernel merges them (log-sum-exp) and normalises.
//  * Every mbarrier wait is bounded; a timeout sets the status word, stops
//    the CTA's producer after its copies in flight have landed, and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "cascade.h"
#include "common.cuh"
#include "mma.cuh"
#include "internal.h"
#include "tmap.h"
#include "prefix.h"

#include <limits.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <type_traits>
#include <vector>

namespace mtkv {
namespace {

constexpr int kMaxConsumerWarps = 8;
constexpr int kThreads = 32 * (kMaxConsumerWarps + 1);
constexpr int kMaxStages = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr unsigned kFull = 0xffffffffu;

enum : int { F_NEW = 1, F_END = 2, F_DATA = 4, F_EXIT = 8 };

struct StageInfo {
  int seq;
  int r0;     // first valid row of the block (relative to the block)
  int r1;     // one past the last valid row
  int flags;  // F_* bits | (first block row held by the stage) << 8
  int mask;   // valid rows of the block as bits (bit t: block row t), within [r0, r1)
};

// Position in the stage ring: slot and the parity of its round, advanced
// without dividing by the (runtime) stage count.
struct RingPos {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void next(int S) {
    if (++slot == (uint32_t)S) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

struct Params {
  CUtensorMap tmap_k;  // tensor-copy path (f16, f32 up to d 128): 3-D maps of the pools, see tma_block()
  CUtensorMap tmap_v;
  const float *q;
  const uint8_t *k_pool;
  const uint8_t *v_pool;
  const int32_t *table;
  const int32_t *ctx;
  const int32_t *spans;
  const int32_t *kv_map;  // [B][MT_KV_MAP_MAX_SPANS][2] (start, len) runs, or null
  float *out;
  float *lse;
  float *part_o;       // [P][Hq][D] unnormalised partial outputs
  float *part_ml;      // [P][Hq][2] partial (max, sum) in base-2 logits
  uint32_t *status;
  const float *k_new;  // [B][Hkv*D] rows appended at position ctx-1, or null
  const float *v_new;
  int B, Hq, Hkv, G, bs, max_blocks;
  long long n_phys;
  int row_bytes;
  int blk_pad;   // bytes of one staged K (or V) row chunk, padded to 128
  int rows;      // block rows per stage (block_size, or a divisor of it for wide rows)
  int pitch;     // shared-memory bytes between consecutive staged rows
  int use_tmap;  // 1: stage blocks with tensor copies (f16 / f32 swizzled, q8_0 padded)
  int pair;      // 1: a stage holds up to two blocks of one sequence (block_size 16, q8_0)
  int scratch_bytes;  // shared-memory bytes between the header and the stage ring
  int ncb;       // 128-byte chunks per staged row (odd), tensor path
  int n_sub;     // partial records per (CTA, sequence) slot
  int stages;
  int wph;       // consumer warps per KV head
  int n_cw;      // consumer warps = Hkv * wph
  int n_ctas;
  float qscale;  // softmax scale * log2(e)
  int combine_wps;  // combine warps per (sequence, query head): 1, 2, 4 or 8
  uint64_t wait_ns;
  Cascade casc;  // shared-prefix groups (n_groups == 0: plain decode)
};

// Shared memory: [barriers | stage infos | abort] header, per-warp softmax
// scratch, then the stage ring.
// shared header: full / empty mbarriers [0, 128), stage records [128, 288),
// the abort flag at 320; scratch from kHdrBytes
constexpr int kHdrBytes = 512;

template <int GP>
__host__ __device__ constexpr int scratch_floats_per_warp() {
  return 32 * GP + GP;  // p[32 tokens][GP] and alpha[GP]
}

// Block rows [a, b) as bits (0 <= a, b <= 32; empty when b <= a).
__device__ __forceinline__ uint32_t row_bits(int a, int b) {
  a = max(a, 0);
  b = min(b, 32);
  if (b <= a) return 0u;
  const uint32_t upto = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
  return upto & ~((1u << a) - 1u);
}

__device__ __forceinline__ int seq_window(const Params &p, int s, int &lo, int &hi) {
  int c = p.ctx[s];
  const int cmax = p.max_blocks * p.bs;
  if (c < 0 || c > cmax) {
    report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
    c = c < 0 ? 0 : cmax;
  }
  lo = 0;
  hi = c;
  if (p.spans) {
    lo = max(p.spans[2 * s], 0);
    hi = min(p.spans[2 * s + 1], c);
  } else if (p.kv_map) {
    // set-valued window: stream the span of its runs; the producer masks
    // the positions between them
    int rl = INT_MAX, rh = INT_MIN;
#pragma unroll
    for (int r = 0; r < MT_KV_MAP_MAX_SPANS; ++r) {
      const int a = max(p.kv_map[((size_t)s * MT_KV_MAP_MAX_SPANS + r) * 2], 0);
      const int e = min(p.kv_map[((size_t)s * MT_KV_MAP_MAX_SPANS + r) * 2] +
                            p.kv_map[((size_t)s * MT_KV_MAP_MAX_SPANS + r) * 2 + 1],
                        c);
      if (e > a) {
        rl = min(rl, a);
        rh = max(rh, e);
      }
    }
    lo = rl;
    hi = rh;
  }
  // cascade: the shared prefix is read by the prefix kernel, not here
  if (p.casc.n_groups) lo = max(lo, cascade_skip(p.casc, s, p.bs));
  if (hi <= lo) {
    lo = hi = 0;
    return 0;
  }
  return (hi - 1) / p.bs - lo / p.bs + 1;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Recursive-halving reduction of N partial sums across the lanes selected by
// offsets OFF, OFF/2, ..., 1: at each of the first log2(N) levels a lane keeps
// the half of its values chosen by its lane bit and adds the partner's copy of
// that half; the remaining levels are plain butterflies. Afterwards acc[0]
// holds the full sum of value index j / (2*OFF/N) (the top log2(N) bits of j).
template <int N, int OFF>
__device__ __forceinline__ void halve(float *acc, int j) {
  if constexpr (OFF > 0) {
    if constexpr (N > 1) {
      const bool upper = (j & OFF) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? acc[i] : acc[i + N / 2];
        const float keep = upper ? acc[i + N / 2] : acc[i];
        acc[i] = keep + __shfl_xor_sync(kFull, send, OFF);
      }
      halve<N / 2, OFF / 2>(acc, j);
    } else {
      acc[0] += __shfl_xor_sync(kFull, acc[0], OFF);
      halve<1, OFF / 2>(acc, j);
    }
  }
}

template <int FMT, int D, int GP>
struct Cfg {
  static constexpr int DPL = (GP >= 8) ? 8 : 16;   // dims per lane in Q.K
  static constexpr int LPT = D / DPL;              // lanes per token
  static constexpr int TPS = 32 / LPT;             // tokens per step
  static constexpr int REP = LPT / GP;             // lanes holding each score
  static constexpr int DV = D / 32;                // P.V dims per lane
  static constexpr int ES = FMT == MT_KV_F32 ? 4 : (FMT == MT_KV_F16 ? 2 : 1);
  static constexpr int CH = FMT == MT_KV_Q8_0 ? DPL : 16 / ES;  // elems per chunk
  static constexpr int NCL = DPL / CH;             // chunks per lane per token
  static constexpr int MAXSTEPS = 32 / TPS;        // steps of a 32-token block
  static_assert(GP <= LPT, "one score per lane");
  static_assert(LPT >= 4 && LPT <= 32, "lane layout");
};

// --------------------------------------------------- swizzled tensor copies
//
// On the f16 tensor-core path a pool is described to the TMA engine as a 3-D
// tensor [cell][128-byte chunk of the row][64 f16], and one tensor copy
// stages `rows` cells of a block with the 128-byte swizzle. The box spans
// ncb chunks, one more than the row has when that count is even (the extra
// chunk lies outside the tensor and is zero-filled, never read from memory),
// so a staged row is an odd number of 128-byte lines: the swizzle then XORs
// the 16-byte unit index with (line & 7) and the 8 rows an ldmatrix phase
// reads land in 8 different bank groups.
__device__ __forceinline__ void tma_block(void *smem_dst, const CUtensorMap *map, int cell,
                                          uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(cell), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// Shared-memory address of the 16-byte unit holding elements [e, e+8) of
// staged row `row` (relative to the stage): line = row*ncb + e/64, unit
// (e/8)%8 XOR (line % 8).
__device__ __forceinline__ uint32_t swz(uint32_t stage, int row, int e, int ncb) {
  const int line = row * ncb + (e >> 6);
  return stage + (uint32_t)line * 128u + ((uint32_t)(((e >> 3) & 7) ^ (line & 7)) << 4);
}

// ------------------------------------------------------------ f16 on MMA
//
// Consumers for f16 pools that run Q.K and P.V on the tensor cores with
// mma.sync.m16n8k16 (f16 inputs, f32 accumulation). Per 16-token step and
// KV head a warp issues 2*(D/16) MMAs for Q.K and D/16 (its share of) MMAs
// for P.V instead of ~1400 FP32-pipe instructions. Layouts:
//   S = Qhl . K^T : A rows r<8 hold the high f16 half of q(head(r)) and rows
//                   r+8 the low half (q - f16(q)), so S = hi + lo is accurate
//                   to ~2^-22 relative; B = K rows straight from shared memory
//                   (ldmatrix); thread (g, c) ends with head(g)'s scores for
//                   tokens 8t + 2c, 8t + 2c + 1.
//   O^T += V^T . P^T : dims on M (ldmatrix.trans of V rows), the N=8 columns
//                   are (head, high/low half of p) pairs when G <= 4 and the
//                   heads themselves when G > 4; each thread supplies column
//                   g from its own probabilities, so P never leaves registers.
// f32 pools take the same path on the same swizzled stages (a row of f32 is
// just more 128-byte lines): K and V values are read as floats and split into
// high / low f16 pairs in registers, and every product runs twice, on the
// high and on the low half (S += Qhl.Khi^T + Qhl.Klo^T, O^T += Vhi^T.P^T +
// Vlo^T.P^T), so scores and outputs keep ~2^-22 relative accuracy.
template <int D, int GP>
struct MmaCfg {
  static constexpr int KS = D / 16;              // Q.K k-steps over the head dims
  static constexpr int MT = D / 16;              // P.V m-tiles over the head dims
  static constexpr int MTW = MT < 8 ? MT : 8;    // m-tiles per warp
  static constexpr int WPH = MT / MTW;           // warps per KV head (split over dims)
  static constexpr bool HILO = GP <= 4;          // p split into two f16 columns
};


// 32-bit shared-memory loads at a shared address
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float2 lds_f32x2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}

// Shared address of float element fe of staged f32 row `row` (same swizzled
// line layout as the f16 rows: element fe is f16 position 2 fe).
__device__ __forceinline__ uint32_t swz32(uint32_t stage, int row, int fe, int ncb) {
  return swz(stage, row, 2 * fe, ncb) + (uint32_t)((fe & 3) * 4);
}

template <int FMT, int D, int GP>
__device__ __forceinline__ void consume_mma(const Params &p, uint64_t *full, uint64_t *empty,
                                            StageInfo *infos, volatile int *abort_flag,
                                            uint8_t *ring, int warp, int lane) {
  using M = MmaCfg<D, GP>;
  const int kvh = warp / M::WPH;
  const int sub = warp % M::WPH;
  const int g = lane >> 2, c = lane & 3;
  const int G = p.G;
  const int S = p.stages;
  const int hrow = M::HILO ? (g >> 1) : g;  // head of A row g (and of B column g)
  const bool row_ok = hrow < G;
  const bool lo_col = M::HILO && (g & 1);   // B column g carries the low half of p
  // lanes holding the softmax state of the heads of O^T columns 2c and 2c+1
  const int src0 = M::HILO ? 8 * c : 8 * c;
  const int src1 = M::HILO ? 8 * c : 8 * c + 4;
  const int head_e = kvh * D;                   // first element of this head in a row
  const int dim0 = sub * M::MTW * 16;           // first output dim of this warp

  uint32_t qa[M::KS][4];
  float oacc[M::MTW][4];
  float m_run = -INFINITY, l_run = 0.f;

  for (RingPos rp;; rp.next(S)) {
    const int slot = (int)rp.slot;
    int okv = 1;
    if (lane == 0)
      okv = mbar_wait_bounded(&full[slot], rp.phase, abort_flag, p.wait_ns) ? 1 : 0;
    okv = __shfl_sync(kFull, okv, 0);
    if (!okv) {
      if (lane == 0) {
        *abort_flag = 1;
        report(p.status, MT_STATUS_BIT_TIMEOUT);
      }
      return;
    }
    int seq, r0, r1, flags, base;
    uint32_t mask;
    {
      const volatile int *vi = reinterpret_cast<const volatile int *>(&infos[slot]);
      seq = vi[0];
      r0 = vi[1];
      r1 = vi[2];
      flags = vi[3] & 0xff;
      base = vi[3] >> 8;
      mask = (uint32_t)vi[4];
    }
    if (flags & F_EXIT) return;

    if (flags & F_NEW) {
      const float *qh = p.q + ((size_t)seq * p.Hq + (size_t)kvh * G + hrow) * D;
#pragma unroll
      for (int ks = 0; ks < M::KS; ++ks) {
        float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
        if (row_ok) {
          x0 = *reinterpret_cast<const float2 *>(qh + 16 * ks + 2 * c);
          x1 = *reinterpret_cast<const float2 *>(qh + 16 * ks + 2 * c + 8);
        }
        split_h2(x0.x * p.qscale, x0.y * p.qscale, qa[ks][0], qa[ks][1]);
        split_h2(x1.x * p.qscale, x1.y * p.qscale, qa[ks][2], qa[ks][3]);
      }
#pragma unroll
      for (int mt = 0; mt < M::MTW; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
    }

    if (flags & F_DATA) {
      const uint32_t kst = smem_u32(ring + (size_t)slot * 2 * p.blk_pad);
      const uint32_t vst = kst + p.blk_pad;
      uint8_t *vst_ptr = ring + (size_t)slot * 2 * p.blk_pad + p.blk_pad;
      const int row_end = base + p.rows;
      // Rows of the stage outside its mask hold bytes of other positions: P
      // is 0 there but 0 * NaN would not be, so clear this head's V chunks of
      // those rows (all 8 units of a chunk, so the swizzle does not matter).
      bool wrote = false;
      const uint32_t bad = row_bits(base, row_end) & ~mask;
      if (bad) {
        constexpr int ES = FMT == MT_KV_F32 ? 4 : 2;
        constexpr int V16 = D * ES / 16;  // 16-byte pieces of one head row
        const int n_bad = __popc(bad);
        for (int i = lane; i < n_bad * V16; i += 32) {
          const int k = i / V16;
          const int row = (int)__fns(bad, 0, k + 1) - base;  // stage row of the k-th bad row
          const int line = row * p.ncb + head_e * ES / 128 + (i % V16) / 8;
          *reinterpret_cast<uint4 *>(vst_ptr + (size_t)line * 128 + (i % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        wrote = true;
        __syncwarp();
      }
      // The stage's NT 8-token tiles (NT = rows / 8, a constant per branch)
      // are all computed, without per-tile conditions, so that their chains
      // interleave: rows outside the stage's mask get score -inf and their V
      // rows are zero (above).
      auto run_stage = [&](auto nt_c) {
      constexpr int NT = decltype(nt_c)::value;
      // ---- S = Qhl . K^T over the stage's 8-token tiles
      float pr[NT][2];
      float mloc = -INFINITY;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int t0 = base + 8 * t;  // block row of the tile's first token
        // two accumulators (alternate products), so the tile's MMAs form two
        // dependent chains of half the length
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, acd[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (FMT == MT_KV_F32) {
          // B fragment of k-step ks: token t0 + g, dims 16 ks + 2c (+1) and + 8
          const int krow = t0 + g - base;
#pragma unroll
          for (int ks = 0; ks < M::KS; ++ks) {
            const int fe = head_e + 16 * ks + 2 * c;
            const float2 k0 = lds_f32x2(swz32(kst, krow, fe, p.ncb));
            const float2 k1 = lds_f32x2(swz32(kst, krow, fe + 8, p.ncb));
            uint32_t h0, l0, h1, l1;
            split_h2(k0.x, k0.y, h0, l0);
            split_h2(k1.x, k1.y, h1, l1);
            mma_f16(acc, qa[ks], h0, h1);
            mma_f16(acd, qa[ks], l0, l1);
          }
        } else {
          const int krow = t0 + (lane & 7) - base;
          const int ke = head_e + ((lane >> 3) & 1) * 8 + (lane >> 4) * 16;
#pragma unroll
          for (int ks = 0; ks < M::KS; ks += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(swz(kst, krow, ke + ks * 16, p.ncb), b0, b1, b2, b3);
            mma_f16(acc, qa[ks], b0, b1);
            mma_f16(acd, qa[ks + 1], b2, b3);
          }
        }
        const int tk = t0 + 2 * c;
        const float s0 = (acc[0] + acd[0]) + (acc[2] + acd[2]);
        const float s1 = (acc[1] + acd[1]) + (acc[3] + acd[3]);
        pr[t][0] = (row_ok && ((mask >> tk) & 1u)) ? s0 : -INFINITY;
        pr[t][1] = (row_ok && ((mask >> (tk + 1)) & 1u)) ? s1 : -INFINITY;
        mloc = fmaxf(mloc, fmaxf(pr[t][0], pr[t][1]));
      }
      // ---- online softmax (base 2) per head: the 4 lanes of group g agree
      mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 1));
      mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 2));
      const float m_new = fmaxf(m_run, mloc);
      const bool none = m_new == -INFINITY;
      const float alpha = none ? 1.f : exp2f(m_run - m_new);
      m_run = m_new;
      float lsum = 0.f;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        pr[t][0] = none ? 0.f : exp2f(pr[t][0] - m_new);
        pr[t][1] = none ? 0.f : exp2f(pr[t][1] - m_new);
        lsum += pr[t][0] + pr[t][1];
      }
      l_run = l_run * alpha + lsum;
      const float a0 = __shfl_sync(kFull, alpha, src0);
      const float a1 = __shfl_sync(kFull, alpha, src1);
      if (!__all_sync(kFull, a0 == 1.f && a1 == 1.f)) {
#pragma unroll
        for (int mt = 0; mt < M::MTW; ++mt) {
          oacc[mt][0] *= a0;
          oacc[mt][1] *= a1;
          oacc[mt][2] *= a0;
          oacc[mt][3] *= a1;
        }
      }
      // ---- O^T += V^T . P^T over 16-token chunks (an 8-row stage, f32 pools
      // with wide rows: one chunk whose tokens 8..15 have P = 0 and V = 0)
      constexpr int NKC = NT >= 2 ? NT / 2 : 1;
#pragma unroll
      for (int kc = 0; kc < NKC; ++kc) {
        const int t0 = base + 16 * kc;
        const float p10 = NT >= 2 ? pr[(2 * kc + 1) % NT][0] : 0.f;
        const float p11 = NT >= 2 ? pr[(2 * kc + 1) % NT][1] : 0.f;
        uint32_t b0, b1;
        if (M::HILO) {
          uint32_t h0, l0, h1, l1;
          split_h2(pr[2 * kc][0], pr[2 * kc][1], h0, l0);
          split_h2(p10, p11, h1, l1);
          b0 = lo_col ? l0 : h0;
          b1 = lo_col ? l1 : h1;
        } else {
          b0 = h2_bits(__floats2half2_rn(pr[2 * kc][0], pr[2 * kc][1]));
          b1 = h2_bits(__floats2half2_rn(p10, p11));
        }
        if (!row_ok) b0 = b1 = 0u;
        if constexpr (FMT == MT_KV_F32) {
          // A = V^T: element (dim g (+8), token 2c (+1) (+8)) read as floats
          const int tr = t0 + 2 * c - base;
#pragma unroll
          for (int mt = 0; mt < M::MTW; ++mt) {
            const int fe = head_e + dim0 + mt * 16 + g;
            float v[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // (dim + 8 (q & 1), token + 8 (q >> 1))
              const int r = tr + 8 * (q >> 1), e = fe + 8 * (q & 1);
              if (NT == 1 && q >= 2) {
                v[2 * q] = v[2 * q + 1] = 0.f;
                continue;
              }
              v[2 * q] = lds_f32(swz32(vst, r, e, p.ncb));
              v[2 * q + 1] = lds_f32(swz32(vst, r + 1, e, p.ncb));
            }
            uint32_t ah[4], al[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) split_h2(v[2 * q], v[2 * q + 1], ah[q], al[q]);
            mma_f16(oacc[mt], ah, b0, b1);
            mma_f16(oacc[mt], al, b0, b1);
          }
        } else {
          const int vrow = t0 + ((lane >> 4) & 1) * 8 + (lane & 7) - base;
          const int ve = head_e + dim0 + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int mt = 0; mt < M::MTW; ++mt) {
            uint32_t a[4];
            ldsm_x4_t(swz(vst, vrow, ve + mt * 16, p.ncb), a[0], a[1], a[2], a[3]);
            mma_f16(oacc[mt], a, b0, b1);
          }
        }
      }
      };
      if constexpr (FMT == MT_KV_F32) {
        if (p.rows == 8) {
          run_stage(std::integral_constant<int, 1>{});
        } else if (p.rows == 16) {
          run_stage(std::integral_constant<int, 2>{});
        } else {
          run_stage(std::integral_constant<int, 4>{});
        }
      } else {
        if (p.rows == 16)
          run_stage(std::integral_constant<int, 2>{});
        else
          run_stage(std::integral_constant<int, 4>{});
      }
      if (wrote) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }

    if (flags & F_END) {
      float l = l_run;
      l += __shfl_xor_sync(kFull, l, 1);
      l += __shfl_xor_sync(kFull, l, 2);
      const size_t P = (size_t)blockIdx.x + seq;
      const size_t hq0 = P * p.Hq + (size_t)kvh * G;
      if (sub == 0 && c == 0 && row_ok && !lo_col) {
        p.part_ml[(hq0 + hrow) * 2 + 0] = m_run;
        p.part_ml[(hq0 + hrow) * 2 + 1] = l;
      }
#pragma unroll
      for (int mt = 0; mt < M::MTW; ++mt) {
        const int dm = dim0 + mt * 16 + g;
        if (M::HILO) {
          if (c < G) {
            float *dst = p.part_o + (hq0 + c) * D;
            dst[dm] = oacc[mt][0] + oacc[mt][1];
            dst[dm + 8] = oacc[mt][2] + oacc[mt][3];
          }
        } else {
          if (2 * c < G) {
            float *dst = p.part_o + (hq0 + 2 * c) * D;
            dst[dm] = oacc[mt][0];
            dst[dm + 8] = oacc[mt][2];
          }
          if (2 * c + 1 < G) {
            float *dst = p.part_o + (hq0 + 2 * c + 1) * D;
            dst[dm] = oacc[mt][1];
            dst[dm + 8] = oacc[mt][3];
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
}

// ----------------------------------------------------------- q8_0 on MMA
//
// q8_0 rows hold 34-byte blocks ({f16 d; int8 q[32]}), so the codes are never
// 16-byte aligned and ldmatrix cannot read them in place. Each consumer warp
// instead converts its head's codes, 16 tokens at a time, into a private f16
// tile in shared memory (exactly: int8 -> f16 by the 1024-bias trick), then
// runs the tensor-core consumer on the tile:
//   S += d[tok][grp] * (Qhl . q^T) per 32-dim group: one accumulator per group
//        and 8-token tile, scaled in f32 by the token's group scale;
//   O^T += q^T . (P * d)^T: the group scale folds into the probability operand
//        (one B fragment per group, hi/lo f16 split), so dequantisation stays
//        exact up to the f16 split of p*d.
// Tile rows are 2*D+16 bytes apart (an odd number of 16-byte units), which
// keeps every ldmatrix phase conflict-free.
//
// A lane converts one 4-code unit in each of its rows: all of its loads are
// issued first, then the conversions and stores, with no branch. Every row
// converts, inside the window or not: q8_0 stages hold 16 or 32 rows and t0 is
// a multiple of 16 inside the stage, so the rows t0 .. t0+15 lie in the
// stage's buffer; int8 codes always give finite f16 values; and a row outside
// the mask gets score -inf and probability 0, so its tile row reaches no
// result.
template <int D>
__device__ __forceinline__ void q8_tile(const uint8_t *st, int row_bytes, int seg, int t0,
                                        uint8_t *tile, int lane) {
  constexpr int GPR = D / 4;      // 4-code units per head row
  constexpr int RPP = 32 / GPR;   // tile rows per warp pass (1 for D = 128, 2 for 64)
  constexpr int NP = 16 / RPP;    // passes over the 16 rows
  constexpr int TP = 2 * D + 16;  // tile pitch in bytes
  const int grp = lane % GPR;
  const int tr = lane / GPR;
  const uint8_t *a = st + (size_t)(t0 + tr) * row_bytes + seg + (grp >> 3) * 34 + 2 + (grp & 7) * 4;
  uint8_t *o = tile + tr * TP + grp * 8;
  uint32_t w[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const uint8_t *ak = a + (size_t)k * RPP * row_bytes;
    const uint32_t lo = *reinterpret_cast<const uint16_t *>(ak);
    const uint32_t hi = *reinterpret_cast<const uint16_t *>(ak + 2);
    w[k] = __byte_perm(lo, hi, 0x5410) ^ 0x80808080u;  // codes + 128, as bytes
  }
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    // f16 bit pattern 0x64XX is 1024 + XX; subtracting 1152 leaves the code
    uint32_t lo = __byte_perm(w[k], 0x64646464u, 0x4140);
    uint32_t hi = __byte_perm(w[k], 0x64646464u, 0x4342);
    lo = h2_bits(__hsub2(*reinterpret_cast<__half2 *>(&lo), bias));
    hi = h2_bits(__hsub2(*reinterpret_cast<__half2 *>(&hi), bias));
    *reinterpret_cast<uint2 *>(o + k * RPP * TP) = make_uint2(lo, hi);
  }
}

__device__ __forceinline__ float q8_scale(const uint8_t *st, int row_bytes, int seg, int tok,
                                          int grp) {
  return __half2float(*reinterpret_cast<const __half *>(st + (size_t)tok * row_bytes + seg +
                                                        grp * 34));
}

// The f32 group scales of rows t0 .. t0+15 of this head, sc[row - t0][group].
// Staged rows sit row_bytes apart (16 banks apart for 1088-byte rows), so the
// fragment lanes that need rows 2c and 2c+1 would all read one bank; from the
// small row-major f32 array they read 4 (or 8) banks apart, without conflict.
// Rows outside the mask may hold any bits here, like their codes: their scores
// are replaced by -inf and their probabilities by 0 before any use.
template <int D>
__device__ __forceinline__ void q8_scales(const uint8_t *st, int row_bytes, int seg, int t0,
                                          float *sc, int lane) {
  constexpr int NG = D / 32;
  constexpr int NP = 16 * NG / 32;  // 2 for D = 128, 1 for 64
  float v[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const int i = lane + 32 * k;
    v[k] = q8_scale(st, row_bytes, seg, t0 + i / NG, i % NG);
  }
#pragma unroll
  for (int k = 0; k < NP; ++k) sc[lane + 32 * k] = v[k];
}

template <int D, int GP>
__device__ __forceinline__ void consume_mma_q8(const Params &p, uint64_t *full, uint64_t *empty,
                                               StageInfo *infos, volatile int *abort_flag,
                                               uint8_t *ring, uint8_t *tiles, int warp,
                                               int lane) {
  using M = MmaCfg<D, GP>;
  static_assert(M::WPH == 1, "q8_0 tensor-core consumers take one warp per KV head");
  constexpr int NG = D / 32;      // q8_0 groups per head
  constexpr int TP = 2 * D + 16;
  const int kvh = warp;
  const int g = lane >> 2, c = lane & 3;
  const int G = p.G;
  const int S = p.stages;
  const int hrow = M::HILO ? (g >> 1) : g;
  const bool row_ok = hrow < G;
  const bool lo_col = M::HILO && (g & 1);
  const int src0 = 8 * c;
  const int src1 = M::HILO ? 8 * c : 8 * c + 4;
  const int seg = kvh * NG * 34;  // byte offset of this head in a row
  uint8_t *tk = tiles + (size_t)warp * 2 * 16 * TP;
  uint8_t *tv = tk + 16 * TP;
  // per-warp f32 group scales of the K and V halves, after all warps' tiles
  float *sk = reinterpret_cast<float *>(tiles + (size_t)kMaxConsumerWarps * 2 * 16 * TP) +
              (size_t)warp * 2 * 16 * NG;
  float *sv = sk + 16 * NG;

  uint32_t qa[M::KS][4];
  float oacc[M::MTW][4];
  float m_run = -INFINITY, l_run = 0.f;

  for (RingPos rp;; rp.next(S)) {
    const int slot = (int)rp.slot;
    int okv = 1;
    if (lane == 0)
      okv = mbar_wait_bounded(&full[slot], rp.phase, abort_flag, p.wait_ns) ? 1 : 0;
    okv = __shfl_sync(kFull, okv, 0);
    if (!okv) {
      if (lane == 0) {
        *abort_flag = 1;
        report(p.status, MT_STATUS_BIT_TIMEOUT);
      }
      return;
    }
    int seq, r0, r1, flags, base;
    uint32_t mask;
    {
      const volatile int *vi = reinterpret_cast<const volatile int *>(&infos[slot]);
      seq = vi[0];
      r0 = vi[1];
      r1 = vi[2];
      flags = vi[3] & 0xff;
      base = vi[3] >> 8;
      mask = (uint32_t)vi[4];
    }
    if (flags & F_EXIT) return;

    if (flags & F_NEW) {
      const float *qh = p.q + ((size_t)seq * p.Hq + (size_t)kvh * G + hrow) * D;
#pragma unroll
      for (int ks = 0; ks < M::KS; ++ks) {
        float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
        if (row_ok) {
          x0 = *reinterpret_cast<const float2 *>(qh + 16 * ks + 2 * c);
          x1 = *reinterpret_cast<const float2 *>(qh + 16 * ks + 2 * c + 8);
        }
        split_h2(x0.x * p.qscale, x0.y * p.qscale, qa[ks][0], qa[ks][1]);
        split_h2(x1.x * p.qscale, x1.y * p.qscale, qa[ks][2], qa[ks][3]);
      }
#pragma unroll
      for (int mt = 0; mt < M::MTW; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
    }

    if (flags & F_DATA) {
      // block-relative rows: stage row r holds block row base + r
      const uint8_t *kst = ring + (size_t)slot * 2 * p.blk_pad - (ptrdiff_t)base * p.row_bytes;
      const uint8_t *vst = kst + p.blk_pad;
      float pr[4][2];
      float mloc = -INFINITY;
      // the first 16-token half's V tile converts together with its K tile,
      // so its loads and stores overlap the K conversion and the scores
      int vh = -1;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t0 = 16 * h;
        pr[2 * h][0] = pr[2 * h][1] = pr[2 * h + 1][0] = pr[2 * h + 1][1] = -INFINITY;
        if (t0 >= p.bs || t0 + 16 <= r0 || t0 >= r1) continue;
        q8_tile<D>(kst, p.row_bytes, seg, t0, tk, lane);
        q8_scales<D>(kst, p.row_bytes, seg, t0, sk, lane);
        if (vh < 0) {
          q8_tile<D>(vst, p.row_bytes, seg, t0, tv, lane);
          q8_scales<D>(vst, p.row_bytes, seg, t0, sv, lane);
          vh = h;
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int tk0 = t0 + 8 * t + 2 * c;
          float s0 = 0.f, s1 = 0.f;
          const uint32_t kaddr = smem_u32(tk + (8 * t + (lane & 7)) * TP) +
                                 (uint32_t)((lane >> 3) & 1) * 16 + (uint32_t)(lane >> 4) * 32;
#pragma unroll
          for (int grp = 0; grp < NG; ++grp) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kaddr + grp * 64, b0, b1, b2, b3);
            mma_f16(acc, qa[2 * grp], b0, b1);
            mma_f16(acc, qa[2 * grp + 1], b2, b3);
            s0 = fmaf(sk[(tk0 - t0) * NG + grp], acc[0] + acc[2], s0);
            s1 = fmaf(sk[(tk0 + 1 - t0) * NG + grp], acc[1] + acc[3], s1);
          }
          pr[2 * h + t][0] = (row_ok && ((mask >> tk0) & 1u)) ? s0 : -INFINITY;
          pr[2 * h + t][1] = (row_ok && ((mask >> (tk0 + 1)) & 1u)) ? s1 : -INFINITY;
          mloc = fmaxf(mloc, fmaxf(pr[2 * h + t][0], pr[2 * h + t][1]));
        }
        __syncwarp();
      }
      // ---- online softmax (base 2), as on the f16 path
      mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 1));
      mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 2));
      const float m_new = fmaxf(m_run, mloc);
      const bool none = m_new == -INFINITY;
      const float alpha = none ? 1.f : exp2f(m_run - m_new);
      m_run = m_new;
      float lsum = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        pr[t][0] = none ? 0.f : exp2f(pr[t][0] - m_new);
        pr[t][1] = none ? 0.f : exp2f(pr[t][1] - m_new);
        lsum += pr[t][0] + pr[t][1];
      }
      l_run = l_run * alpha + lsum;
      const float a0 = __shfl_sync(kFull, alpha, src0);
      const float a1 = __shfl_sync(kFull, alpha, src1);
      if (!__all_sync(kFull, a0 == 1.f && a1 == 1.f)) {
#pragma unroll
        for (int mt = 0; mt < M::MTW; ++mt) {
          oacc[mt][0] *= a0;
          oacc[mt][1] *= a1;
          oacc[mt][2] *= a0;
          oacc[mt][3] *= a1;
        }
      }
      // ---- O^T += q^T . (P * d)^T per 16-token half
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t0 = 16 * h;
        if (t0 >= p.bs || t0 + 16 <= r0 || t0 >= r1) continue;
        if (h != vh) {
          q8_tile<D>(vst, p.row_bytes, seg, t0, tv, lane);
          q8_scales<D>(vst, p.row_bytes, seg, t0, sv, lane);
          __syncwarp();
        }
        const uint32_t vaddr = smem_u32(tv + (((lane >> 4) & 1) * 8 + (lane & 7)) * TP) +
                               (uint32_t)((lane >> 3) & 1) * 16;
        const int ta = t0 + 2 * c, tb = t0 + 8 + 2 * c;  // this thread's B rows (tokens)
        const bool va0 = (mask >> ta) & 1u, va1 = (mask >> (ta + 1)) & 1u;
        const bool vb0 = (mask >> tb) & 1u, vb1 = (mask >> (tb + 1)) & 1u;
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) {
          const float pa0 = va0 ? pr[2 * h][0] * sv[(ta - t0) * NG + grp] : 0.f;
          const float pa1 = va1 ? pr[2 * h][1] * sv[(ta + 1 - t0) * NG + grp] : 0.f;
          const float pb0 = vb0 ? pr[2 * h + 1][0] * sv[(tb - t0) * NG + grp] : 0.f;
          const float pb1 = vb1 ? pr[2 * h + 1][1] * sv[(tb + 1 - t0) * NG + grp] : 0.f;
          uint32_t bq0, bq1;
          if (M::HILO) {
            uint32_t h0, l0, h1, l1;
            split_h2(pa0, pa1, h0, l0);
            split_h2(pb0, pb1, h1, l1);
            bq0 = lo_col ? l0 : h0;
            bq1 = lo_col ? l1 : h1;
          } else {
            bq0 = h2_bits(__floats2half2_rn(pa0, pa1));
            bq1 = h2_bits(__floats2half2_rn(pb0, pb1));
          }
          if (!row_ok) bq0 = bq1 = 0u;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int mt = 2 * grp + j;
            uint32_t a[4];
            ldsm_x4_t(vaddr + mt * 32, a[0], a[1], a[2], a[3]);
            mma_f16(oacc[mt], a, bq0, bq1);
          }
        }
        __syncwarp();
      }
    }

    if (flags & F_END) {
      float l = l_run;
      l += __shfl_xor_sync(kFull, l, 1);
      l += __shfl_xor_sync(kFull, l, 2);
      const size_t P = (size_t)blockIdx.x + seq;
      const size_t hq0 = P * p.Hq + (size_t)kvh * G;
      if (c == 0 && row_ok && !lo_col) {
        p.part_ml[(hq0 + hrow) * 2 + 0] = m_run;
        p.part_ml[(hq0 + hrow) * 2 + 1] = l;
      }
#pragma unroll
      for (int mt = 0; mt < M::MTW; ++mt) {
        const int dm = mt * 16 + g;
        if (M::HILO) {
          if (c < G) {
            float *dst = p.part_o + (hq0 + c) * D;
            dst[dm] = oacc[mt][0] + oacc[mt][1];
            dst[dm + 8] = oacc[mt][2] + oacc[mt][3];
          }
        } else {
          if (2 * c < G) {
            float *dst = p.part_o + (hq0 + 2 * c) * D;
            dst[dm] = oacc[mt][0];
            dst[dm + 8] = oacc[mt][2];
          }
          if (2 * c + 1 < G) {
            float *dst = p.part_o + (hq0 + 2 * c + 1) * D;
            dst[dm] = oacc[mt][1];
            dst[dm + 8] = oacc[mt][3];
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
}

// ------------------------------------ q8_0 on MMA, operands from the rows
//
// For head_dim 128 the q8_0 consumer builds its tensor-core operands
// straight from the staged rows instead of converting whole code tiles
// through shared memory (no tile stores, no ldmatrix, no warp barrier
// between conversion and use):
//   * S = Q.K^T per 32-dim group: inside a group, the k-slots (2c, 2c+1,
//     2c+8, 2c+9) of k-step j stand for dims 8c + 4j + (0, 1, 2, 3). Lane
//     (g, c) of the B operand then needs the 8 consecutive codes [8c, 8c+8)
//     of its token: one or two loads from the staged row, because a group's
//     codes start 2 bytes after its f16 scale at an offset whose residue
//     mod 8 is fixed (rows and head segments are whole 8-byte units for
//     head_dim 128). Q's A fragments are built in the same dim order.
//   * O^T += V^T.(P*d)^T: the A-operand rows of a group's two 16-dim m-tiles
//     stand for dims 4g + (0, 1) and 4g + (2, 3), so lane (g, c) loads one
//     4-code word per token and pairs two tokens' words with byte permutes
//     (a register of the A operand holds two k-slots, i.e. two tokens, of
//     one dim).
//   * The score columns of a 16-row half take its tokens in the order
//     0 4 1 5 2 6 3 7 | 8 12 9 13 10 14 11 15, so the four tokens a lane holds
//     probabilities for (c, 4+c, 8+c, 12+c) are exactly the four k-slots it
//     supplies to P.V: P never leaves registers.
// int8 -> f16 is exact (the 1024-bias byte permute); each half's group
// scales are read once into two small f32 arrays in score-column order.
// Every row of a half converts, valid or not: codes always give finite
// values, and an invalid row gets score -inf and a zero P.V operand (its
// scale, which may be stale bits, is never multiplied in).

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void lds_u32x2(uint32_t a, uint32_t &x, uint32_t &y) {
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(a));
}
__device__ __forceinline__ float lds_f16f(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return __half2float(__ushort_as_half(v));
}

// The 8 bytes at shared address a, where a % 8 == MIS (even): x = bytes
// [a, a+4), y = bytes [a+4, a+8), with aligned loads only.
template <int MIS>
__device__ __forceinline__ void lds_code8(uint32_t a, uint32_t &x, uint32_t &y) {
  static_assert(MIS == 0 || MIS == 2 || MIS == 4 || MIS == 6, "even offset");
  if constexpr (MIS == 0) {
    lds_u32x2(a, x, y);
  } else if constexpr (MIS == 4) {
    x = lds_u32(a);
    y = lds_u32(a + 4);
  } else if constexpr (MIS == 2) {
    uint32_t w0, w1;
    lds_u32x2(a - 2, w0, w1);
    const uint32_t w2 = lds_u32(a + 6);
    x = __byte_perm(w0, w1, 0x5432);
    y = __byte_perm(w1, w2, 0x5432);
  } else {
    const uint32_t w0 = lds_u32(a - 2);
    uint32_t w1, w2;
    lds_u32x2(a + 2, w1, w2);
    x = __byte_perm(w0, w1, 0x5432);
    y = __byte_perm(w1, w2, 0x5432);
  }
}

// The 4 bytes at shared address a, a % 4 == MIS (0 or 2).
template <int MIS>
__device__ __forceinline__ uint32_t lds_code4(uint32_t a) {
  if constexpr (MIS == 0) {
    return lds_u32(a);
  } else {
    return __byte_perm(lds_u32(a - 2), lds_u32(a + 2), 0x5432);
  }
}

// f16 bit patterns 0x64XX are 1024 + XX: codes + 128 as bytes, then minus 1152
__device__ __forceinline__ uint32_t biased_to_h2(uint32_t b, uint32_t sel) {
  uint32_t h = __byte_perm(b, 0x64646464u, sel);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  return h2_bits(__hsub2(*reinterpret_cast<__half2 *>(&h), bias));
}

// int8 codes of word w (bytes 0..3) -> f16 pairs (code0, code1), (code2, code3)
__device__ __forceinline__ void codes_to_h2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t b = w ^ 0x80808080u;
  lo = biased_to_h2(b, 0x4140);
  hi = biased_to_h2(b, 0x4342);
}

// words x (one token's codes of dims k..k+3) and y (another token's, same
// dims) -> f16 pairs (x_i, y_i) for i = 0..3
__device__ __forceinline__ void code_pairs_to_h2(uint32_t x, uint32_t y, uint32_t (&o)[4]) {
  const uint32_t lo = __byte_perm(x, y, 0x5140) ^ 0x80808080u;  // x0 y0 x1 y1
  const uint32_t hi = __byte_perm(x, y, 0x7362) ^ 0x80808080u;  // x2 y2 x3 y3
  o[0] = biased_to_h2(lo, 0x4140);
  o[1] = biased_to_h2(lo, 0x4342);
  o[2] = biased_to_h2(hi, 0x4140);
  o[3] = biased_to_h2(hi, 0x4342);
}

// Token (row within a 16-row half) of score column position pos = 8t + n.
__host__ __device__ constexpr int q8d_col_token(int pos) {
  return 8 * (pos >> 3) + ((pos & 7) >> 1) + 4 * (pos & 1);
}

// mma with a zero accumulator input: d = a.b
__device__ __forceinline__ void mma_f16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// Per-warp f32 scale arrays of the direct q8_0 consumer: K and V, for each
// 16-row half of a stage, [group][score-column position].
constexpr int kQ8dScaleFloatsPerHalf = 2 * 4 * 16;

template <int GP, int NH>
__device__ __forceinline__ void consume_q8_direct(const Params &p, uint64_t *full,
                                                  uint64_t *empty, StageInfo *infos,
                                                  volatile int *abort_flag, uint8_t *ring,
                                                  float *scr, int warp, int lane) {
  constexpr int D = 128;
  constexpr int NG = 4;                 // q8_0 groups per head
  constexpr bool HILO = GP <= 4;        // p split into two f16 columns
  const int kvh = warp;
  const int g = lane >> 2, c = lane & 3;
  const int G = p.G;
  const int S = p.stages;
  const int hrow = HILO ? (g >> 1) : g;
  const bool row_ok = hrow < G;
  const bool lo_col = HILO && (g & 1);
  const int src0 = 8 * c;
  const int src1 = HILO ? 8 * c : 8 * c + 4;
  const uint32_t seg = (uint32_t)kvh * (NG * 34);  // this head's bytes in a row
  const uint32_t pitch = (uint32_t)p.pitch;
  float *sK = scr + (size_t)warp * (NH * kQ8dScaleFloatsPerHalf);  // [h][grp][16]
  float *sV = sK + NH * NG * 16;
  // this lane's K row within a 16-row half (tile t adds 8): score column g
  const int krow = (g >> 1) + 4 * (g & 1);
  const uint32_t ring_s = smem_u32(ring);

  uint32_t qa[NG][2][4];
  float oacc[2 * NG][4];
  float m_run = -INFINITY, l_run = 0.f;

  for (RingPos rp;; rp.next(S)) {
    const int slot = (int)rp.slot;
    int okv = 1;
    if (lane == 0)
      okv = mbar_wait_bounded(&full[slot], rp.phase, abort_flag, p.wait_ns) ? 1 : 0;
    okv = __shfl_sync(kFull, okv, 0);
    if (!okv) {
      if (lane == 0) {
        *abort_flag = 1;
        report(p.status, MT_STATUS_BIT_TIMEOUT);
      }
      return;
    }
    int seq, flags, base;
    uint32_t mask;
    {
      const volatile int *vi = reinterpret_cast<const volatile int *>(&infos[slot]);
      seq = vi[0];
      flags = vi[3] & 0xff;
      base = vi[3] >> 8;
      mask = (uint32_t)vi[4];
    }
    if (flags & F_EXIT) return;

    if (flags & F_NEW) {
      const float *qh = p.q + ((size_t)seq * p.Hq + (size_t)kvh * G + hrow) * D;
#pragma unroll
      for (int grp = 0; grp < NG; ++grp)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row_ok) x = *reinterpret_cast<const float4 *>(qh + 32 * grp + 8 * c + 4 * j);
          split_h2(x.x * p.qscale, x.y * p.qscale, qa[grp][j][0], qa[grp][j][1]);
          split_h2(x.z * p.qscale, x.w * p.qscale, qa[grp][j][2], qa[grp][j][3]);
        }
#pragma unroll
      for (int mt = 0; mt < 2 * NG; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
    }

    if (flags & F_DATA) {
      const uint32_t kst = ring_s + (uint32_t)slot * 2u * (uint32_t)p.blk_pad;
      const uint32_t vst = kst + (uint32_t)p.blk_pad;
      // ---- group scales of both pools, per half, in score-column order; a V
      // scale of a row outside the mask is stored as 0 (its bits may be stale)
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const uint32_t mh = (mask >> (base + 16 * h)) & 0xffffu;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int i = lane + 32 * k;          // [grp][pos]
          const int grp = i >> 4, pos = i & 15;
          const int tok = q8d_col_token(pos);
          const uint32_t off = (uint32_t)(16 * h + tok) * pitch + seg + 34u * grp;
          const float dk = lds_f16f(kst + off);
          const float dv = lds_f16f(vst + off);
          sK[h * NG * 16 + i] = dk;
          sV[h * NG * 16 + i] = ((mh >> tok) & 1u) ? dv : 0.f;
        }
      }
      // ---- every K code word of the stage, loaded before any conversion
      uint32_t w[NH][2][NG][2];
#pragma unroll
      for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t ka = kst + (uint32_t)(16 * h + 8 * t + krow) * pitch + seg + 2u + 8u * c;
          lds_code8<2>(ka, w[h][t][0][0], w[h][t][0][1]);
          lds_code8<4>(ka + 34, w[h][t][1][0], w[h][t][1][1]);
          lds_code8<6>(ka + 68, w[h][t][2][0], w[h][t][2][1]);
          lds_code8<0>(ka + 102, w[h][t][3][0], w[h][t][3][1]);
        }
      __syncwarp();
      // ---- scores: two 8-column tiles per half
      float pr[NH][2][2];
      float mloc = -INFINITY;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const uint32_t mh = (mask >> (base + 16 * h)) & 0xffffu;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          float2 sv2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int grp = 0; grp < NG; ++grp) {
            uint32_t b[2][2];
            codes_to_h2(w[h][t][grp][0], b[0][0], b[0][1]);
            codes_to_h2(w[h][t][grp][1], b[1][0], b[1][1]);
            float acc[4];
            mma_f16_z(acc, qa[grp][0], b[0][0], b[0][1]);
            mma_f16(acc, qa[grp][1], b[1][0], b[1][1]);
            const float2 sc = *reinterpret_cast<const float2 *>(sK + h * NG * 16 + grp * 16 +
                                                                8 * t + 2 * c);
            // (hi + lo rows) times the tokens' group scales, two tokens at once
            sv2 = f2_fma(sc, f2_add(make_float2(acc[0], acc[1]), make_float2(acc[2], acc[3])), sv2);
          }
          const bool v0 = row_ok && ((mh >> (8 * t + c)) & 1u);
          const bool v1 = row_ok && ((mh >> (8 * t + 4 + c)) & 1u);
          pr[h][t][0] = v0 ? sv2.x : -INFINITY;
          pr[h][t][1] = v1 ? sv2.y : -INFINITY;
          mloc = fmaxf(mloc, fmaxf(pr[h][t][0], pr[h][t][1]));
        }
      }
      // ---- the V code words of the first half, loaded before the softmax
      // (the k-slots 2c, 2c+1, 2c+8, 2c+9 are tokens c, 4+c, 8+c, 12+c)
      const uint32_t p4 = 4u * pitch;
      uint32_t wv[NG][4];
      const uint32_t va0 = vst + (uint32_t)c * pitch + seg + 2u + 4u * g;
      {
        const uint32_t vr[4] = {va0, va0 + p4, va0 + 2 * p4, va0 + 3 * p4};
#pragma unroll
        for (int grp = 0; grp < NG; ++grp)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            wv[grp][k] = (grp & 1) ? lds_code4<0>(vr[k] + 34u * grp) : lds_code4<2>(vr[k] + 34u * grp);
      }
      // ---- online softmax (base 2); a lane's tokens of a half are c, 4+c,
      // 8+c, 12+c, the group's four lanes cover all sixteen
      mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 1));
      mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 2));
      const float m_new = fmaxf(m_run, mloc);
      const bool none = m_new == -INFINITY;
      const float alpha = none ? 1.f : exp2f(m_run - m_new);
      m_run = m_new;
      float lsum = 0.f;
#pragma unroll
      for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          pr[h][t][0] = none ? 0.f : exp2f(pr[h][t][0] - m_new);
          pr[h][t][1] = none ? 0.f : exp2f(pr[h][t][1] - m_new);
          lsum += pr[h][t][0] + pr[h][t][1];
        }
      l_run = l_run * alpha + lsum;
      const float a0 = __shfl_sync(kFull, alpha, src0);
      const float a1 = __shfl_sync(kFull, alpha, src1);
      if (!__all_sync(kFull, a0 == 1.f && a1 == 1.f)) {
#pragma unroll
        for (int mt = 0; mt < 2 * NG; ++mt) {
          oacc[mt][0] *= a0;
          oacc[mt][1] *= a1;
          oacc[mt][2] *= a0;
          oacc[mt][3] *= a1;
        }
      }
      // ---- O^T += V^T . (P * d)^T, per half and group
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        if (h > 0) {
          const uint32_t va = va0 + (uint32_t)(16 * h) * pitch;
          const uint32_t vr[4] = {va, va + p4, va + 2 * p4, va + 3 * p4};
#pragma unroll
          for (int grp = 0; grp < NG; ++grp)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              wv[grp][k] = (grp & 1) ? lds_code4<0>(vr[k] + 34u * grp) : lds_code4<2>(vr[k] + 34u * grp);
        }
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) {
          uint32_t o01[4], o23[4];
          code_pairs_to_h2(wv[grp][0], wv[grp][1], o01);
          code_pairs_to_h2(wv[grp][2], wv[grp][3], o23);
          // V scales of rows outside the mask are 0 and their p is 0
          const float *sv = sV + h * NG * 16 + grp * 16;
          const float2 s01 = *reinterpret_cast<const float2 *>(sv + 2 * c);
          const float2 s23 = *reinterpret_cast<const float2 *>(sv + 8 + 2 * c);
          const float2 pa = f2_mul(make_float2(pr[h][0][0], pr[h][0][1]), s01);
          const float2 pb = f2_mul(make_float2(pr[h][1][0], pr[h][1][1]), s23);
          uint32_t bq0, bq1;
          if (HILO) {
            uint32_t h0, l0, h1, l1;
            split_h2x(pa, h0, l0);
            split_h2x(pb, h1, l1);
            bq0 = lo_col ? l0 : h0;
            bq1 = lo_col ? l1 : h1;
          } else {
            bq0 = h2_bits(__floats2half2_rn(pa.x, pa.y));
            bq1 = h2_bits(__floats2half2_rn(pb.x, pb.y));
          }
          if (!row_ok) bq0 = bq1 = 0u;
          const uint32_t am0[4] = {o01[0], o01[1], o23[0], o23[1]};  // dims 4g, 4g+1
          const uint32_t am1[4] = {o01[2], o01[3], o23[2], o23[3]};  // dims 4g+2, 4g+3
          mma_f16(oacc[2 * grp], am0, bq0, bq1);
          mma_f16(oacc[2 * grp + 1], am1, bq0, bq1);
        }
      }
    }

    if (flags & F_END) {
      float l = l_run;
      l += __shfl_xor_sync(kFull, l, 1);
      l += __shfl_xor_sync(kFull, l, 2);
      const size_t P = (size_t)blockIdx.x + seq;
      const size_t hq0 = P * p.Hq + (size_t)kvh * G;
      if (c == 0 && row_ok && !lo_col) {
        p.part_ml[(hq0 + hrow) * 2 + 0] = m_run;
        p.part_ml[(hq0 + hrow) * 2 + 1] = l;
      }
      // rows g, g+8 of m-tiles 2grp, 2grp+1 are dims 32grp + 4g + (0, 1, 2, 3)
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        const float *o0 = oacc[2 * grp], *o1 = oacc[2 * grp + 1];
        if (HILO) {
          if (c < G)
            *reinterpret_cast<float4 *>(p.part_o + (hq0 + c) * D + 32 * grp + 4 * g) =
                make_float4(o0[0] + o0[1], o0[2] + o0[3], o1[0] + o1[1], o1[2] + o1[3]);
        } else {
          if (2 * c < G)
            *reinterpret_cast<float4 *>(p.part_o + (hq0 + 2 * c) * D + 32 * grp + 4 * g) =
                make_float4(o0[0], o0[2], o1[0], o1[2]);
          if (2 * c + 1 < G)
            *reinterpret_cast<float4 *>(p.part_o + (hq0 + 2 * c + 1) * D + 32 * grp + 4 * g) =
                make_float4(o0[1], o0[3], o1[1], o1[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
}

// Fused store of one sequence's new row (decode with append): convert
// k_new[s] and v_new[s] to the pool format and write them into `cell` of
// both pools, by the 32 lanes of the calling warp, with the arithmetic of
// kv_store_kernel (so the bytes are the same). Loads go out in batches of 8
// per lane before any store. Ends with each lane's proxy fence and a warp
// barrier: a bulk copy issued afterwards by any lane reads the new bytes.
template <int FMT, int D>
__device__ __noinline__ void append_row(const Params &p, int s, long long cell, int lane) {
  const int n = p.Hkv * D;
#pragma unroll 1
  for (int kv = 0; kv < 2; ++kv) {
    const float *src = (kv ? p.v_new : p.k_new) + (size_t)s * n;
    uint8_t *dst = const_cast<uint8_t *>(kv ? p.v_pool : p.k_pool) + (size_t)cell * p.row_bytes;
    if constexpr (FMT == MT_KV_Q8_0) {
      const int groups = n / 32;
#pragma unroll 1
      for (int g0 = 0; g0 < groups; g0 += 8) {
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = g0 + j < groups ? src[(g0 + j) * 32 + lane] : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (g0 + j < groups) q8_quant_group(dst + (size_t)(g0 + j) * 34, x[j], lane);
      }
      const int pad = p.row_bytes - groups * 34;
      if (lane < pad) dst[groups * 34 + lane] = 0;
    } else {
#pragma unroll 1
      for (int i0 = 4 * lane; i0 < n; i0 += 128 * 8) {
        float4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + 128 * j;
          x[j] = i < n ? *reinterpret_cast<const float4 *>(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + 128 * j;
          if (i >= n) break;
          if constexpr (FMT == MT_KV_F32) {
            *reinterpret_cast<float4 *>(dst + (size_t)i * 4) = x[j];
          } else {
            const __half2 a = __floats2half2_rn(x[j].x, x[j].y);
            const __half2 b = __floats2half2_rn(x[j].z, x[j].w);
            *reinterpret_cast<uint2 *>(dst + (size_t)i * 2) =
                make_uint2(*reinterpret_cast<const uint32_t *>(&a),
                           *reinterpret_cast<const uint32_t *>(&b));
          }
        }
      }
    }
  }
  fence_proxy_async_global();
  __syncwarp();
}

// Set-valued window: the rows of logical block lb of sequence s that one of
// its (start, len) runs covers, within the sequence's window [lo, hi); lane r
// of the calling warp takes run r. Kept out of line: only kv_map calls pay.
__device__ __noinline__ uint32_t kv_map_block_mask(const Params &p, int s, int lb, int lo, int hi,
                                                   int lane) {
  uint32_t m = 0u;
  if (lane < MT_KV_MAP_MAX_SPANS) {
    const int32_t *rp = p.kv_map + ((size_t)s * MT_KV_MAP_MAX_SPANS + lane) * 2;
    const int a = max(rp[0], lo), e = min(rp[0] + rp[1], hi);
    m = row_bits(a - lb * p.bs, e - lb * p.bs);
  }
  return __reduce_or_sync(kFull, m);
}

// Part `part` of `n_parts` of the work of append_row (q8_0: 32-value groups
// part, part + n_parts, ...; f16/f32: 4-value chunks likewise), for rows that
// no CTA reads in this launch, so no ordering with any copy is needed.
template <int FMT, int D>
__device__ __noinline__ void append_row_part(const Params &p, int s, long long cell, int lane,
                                             int part, int n_parts) {
  const int n = p.Hkv * D;
#pragma unroll 1
  for (int kv = 0; kv < 2; ++kv) {
    const float *src = (kv ? p.v_new : p.k_new) + (size_t)s * n;
    uint8_t *dst = const_cast<uint8_t *>(kv ? p.v_pool : p.k_pool) + (size_t)cell * p.row_bytes;
    if constexpr (FMT == MT_KV_Q8_0) {
      const int groups = n / 32;
#pragma unroll 1
      for (int g = part; g < groups; g += n_parts)
        q8_quant_group(dst + (size_t)g * 34, src[g * 32 + lane], lane);
      const int pad = p.row_bytes - groups * 34;
      if (part == 0 && lane < pad) dst[groups * 34 + lane] = 0;
    } else {
#pragma unroll 1
      for (int i = 4 * lane + 128 * part; i < n; i += 128 * n_parts) {
        const float4 x = *reinterpret_cast<const float4 *>(src + i);
        if constexpr (FMT == MT_KV_F32) {
          *reinterpret_cast<float4 *>(dst + (size_t)i * 4) = x;
        } else {
          const __half2 a = __floats2half2_rn(x.x, x.y);
          const __half2 b = __floats2half2_rn(x.z, x.w);
          *reinterpret_cast<uint2 *>(dst + (size_t)i * 2) =
              make_uint2(*reinterpret_cast<const uint32_t *>(&a),
                         *reinterpret_cast<const uint32_t *>(&b));
        }
      }
    }
  }
}

// Position ctx-1 of sequence s, for decode with append: its logical block,
// or -1 when the context length is out of range (flagged) or zero.
__device__ __forceinline__ int append_block(const Params &p, int s) {
  const int c = p.ctx[s];
  if (c <= 0 || c > p.max_blocks * p.bs) return -1;
  return (c - 1) / p.bs;
}

// MINB: CTAs per SM the kernel is compiled for (2 only for the direct q8_0
// consumer with 16-row stages, whose registers then fit two resident CTAs).
template <int FMT, int D, int GP, bool MMA, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    paged_decode_kernel(const __grid_constant__ Params p) {
  using C = Cfg<FMT, D, GP>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + kMaxStages;
  StageInfo *infos = reinterpret_cast<StageInfo *>(smem + 128);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 320);
  float *scratch = reinterpret_cast<float *>(smem + kHdrBytes);
  // the ring starts on a 1024-byte boundary (the 128-byte swizzle's period)
  uint8_t *ring = smem + kHdrBytes + p.scratch_bytes;
  ring += (1024u - (smem_u32(ring) & 1023u)) & 1023u;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  // the successor may start launching at once; every role waits for the
  // predecessor (pdl_wait) before its first access to memory an earlier
  // kernel of the stream may write: the producer first plans its range from
  // the context lengths, windows and block table, which no kernel of this
  // library writes, so that work overlaps the predecessor's tail
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], p.n_cw);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == p.n_cw) {
    // ------------------------------------------------------ producer warp
    const uint64_t pol = policy_evict_first();
    // pass 1: total stream length
    int total = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int s = base + lane;
      int lo, hi;
      const int nb = s < p.B ? seq_window(p, s, lo, hi) : 0;
      const int incl = warp_incl_scan(nb, lane);
      total += __shfl_sync(kFull, incl, 31);
    }
    const int per = total > 0 ? (total + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    const long long b0 = (long long)blockIdx.x * per;
    const long long b1 = min((long long)total, b0 + per);

    uint32_t it = 0;
    RingPos prp;  // slot and round parity of stage `it`
    bool alive = true;
    // Publish one stage. Lane 0 waits for the slot and issues; the others
    // learn the outcome through the shuffle.
    auto emit = [&](int flags, int s, int r0, int r1, int phys, int base, uint32_t mask,
                    int phys2 = -1) -> bool {
      const int slot = (int)prp.slot;
      int okv = 1;
      if (lane == 0) {
        // the slot's previous fill (round - 1) must have been released
        if (it >= (uint32_t)S && !mbar_wait_bounded(&empty[slot], prp.phase ^ 1u, abort_flag,
                                                    p.wait_ns))
          okv = 0;
        if (okv) {
          infos[slot] = StageInfo{s, r0, r1, flags | (base << 8), (int)mask};
          if ((flags & F_DATA) && p.pair) {
            // block phys in rows [0, bs), block phys2 (if any) in [bs, 2 bs):
            // one tensor copy per block and pool
            uint8_t *dk = ring + (size_t)slot * 2 * p.blk_pad;
            const uint32_t half = (uint32_t)(p.bs * p.pitch);
            mbar_arrive_expect_tx(&full[slot], (phys2 >= 0 ? 4u : 2u) * half);
            tma_block(dk, &p.tmap_k, phys * p.bs, &full[slot], pol);
            tma_block(dk + p.blk_pad, &p.tmap_v, phys * p.bs, &full[slot], pol);
            if (phys2 >= 0) {
              tma_block(dk + half, &p.tmap_k, phys2 * p.bs, &full[slot], pol);
              tma_block(dk + p.blk_pad + half, &p.tmap_v, phys2 * p.bs, &full[slot], pol);
            }
          } else if ((flags & F_DATA) && p.use_tmap) {
            // the whole stage (rows [base, base + rows)) in two tensor copies
            uint8_t *dk = ring + (size_t)slot * 2 * p.blk_pad;
            const int cell = phys * p.bs + base;
            mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * p.rows * p.pitch));
            tma_block(dk, &p.tmap_k, cell, &full[slot], pol);
            tma_block(dk + p.blk_pad, &p.tmap_v, cell, &full[slot], pol);
          } else if (flags & F_DATA) {
            // rows [ra, rb): the valid rows widened to whole 4-row groups, so
            // both addresses and the size stay multiples of 16 bytes
            const int ra = r0 & ~3;
            const int rb = min(base + p.rows, (r1 + 3) & ~3);
            const uint32_t bytes = (uint32_t)((rb - ra) * p.row_bytes);
            uint8_t *dk = ring + (size_t)slot * 2 * p.blk_pad + (size_t)(ra - base) * p.row_bytes;
            const size_t src = ((size_t)phys * p.bs + ra) * (size_t)p.row_bytes;
            mbar_arrive_expect_tx(&full[slot], 2 * bytes);
            bulk_g2s(dk, p.k_pool + src, bytes, &full[slot], pol);
            bulk_g2s(dk + p.blk_pad, p.v_pool + src, bytes, &full[slot], pol);
          } else {
            mbar_arrive(&full[slot]);
          }
        }
      }
      okv = __shfl_sync(kFull, okv, 0);
      if (okv) {
        ++it;
        prp.next(S);
      }
      return okv != 0;
    };

    // pass 2: first sequence whose blocks reach past b0
    int s_first = p.B, start_first = 0;
    if (b0 < b1) {
      int run = 0;
      for (int base = 0; base < p.B; base += 32) {
        const int s = base + lane;
        int lo, hi;
        const int nb = s < p.B ? seq_window(p, s, lo, hi) : 0;
        const int incl = warp_incl_scan(nb, lane);
        const unsigned hit = __ballot_sync(kFull, s < p.B && nb > 0 && (long long)run + incl > b0);
        if (hit) {
          const int l = __ffs(hit) - 1;
          s_first = base + l;
          start_first = run + __shfl_sync(kFull, incl - nb, l);
          break;
        }
        run += __shfl_sync(kFull, incl, 31);
      }
    }
    pdl_wait();
    if (b0 < b1) {
      long long x = b0;
      int start = start_first;
      for (int s = s_first; alive && x < b1 && s < p.B; ++s) {
        int lo, hi;
        const int nb = seq_window(p, s, lo, hi);
        const long long seg_lo = max(x, (long long)start);
        const long long seg_hi = min(b1, (long long)start + nb);
        if (seg_hi > seg_lo) {
          if (lane == 0)
            bulk_prefetch_l2(p.q + (size_t)s * p.Hq * D, (uint32_t)(p.Hq * D * sizeof(float)));
          bool first = true;
          int pend = -1;           // paired stages: block waiting for its partner
          uint32_t pend_mask = 0;
          const int lb0 = lo / p.bs;
          // decode with append: the logical block of position ctx-1 when this
          // segment loads it (its new row is written just before the copy)
          int lb_app = -1;
          if (p.k_new) {
            const int lb = append_block(p, s);
            if (lb >= lb0 + (int)(seg_lo - start) && lb < lb0 + (int)(seg_hi - start)) {
              lb_app = lb;
              if (lane == 0) {
                const uint32_t row = (uint32_t)(p.Hkv * D * sizeof(float));
                bulk_prefetch_l2(p.k_new + (size_t)s * p.Hkv * D, row);
                bulk_prefetch_l2(p.v_new + (size_t)s * p.Hkv * D, row);
              }
            }
          }
          const int32_t *trow = p.table + (size_t)s * p.max_blocks;
          for (long long y0 = seg_lo; alive && y0 < seg_hi; y0 += 32) {
            const long long y = y0 + lane;
            int ent = MT_INVALID_BLOCK_ID;
            if (y < seg_hi) ent = trow[lb0 + (int)(y - start)];
            const int cnt = (int)min(32LL, seg_hi - y0);
            for (int i = 0; i < cnt; ++i) {
              const int phys = __shfl_sync(kFull, ent, i);
              const int lb = lb0 + (int)(y0 + i - start);
              if (lb == lb_app) {
                if (phys < 0 || (long long)phys >= p.n_phys) {
                  if (lane == 0) report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
                } else {
                  append_row<FMT, D>(p, s, (long long)phys * p.bs + (p.ctx[s] - 1) % p.bs, lane);
                }
              }
              if (phys == MT_INVALID_BLOCK_ID) continue;
              if (phys < 0 || (long long)phys >= p.n_phys) {
                if (lane == 0) report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
                continue;
              }
              const int r0 = max(lo - lb * p.bs, 0);
              const int r1 = min(hi - lb * p.bs, p.bs);
              uint32_t bmask = row_bits(r0, r1);
              if (p.kv_map) {
                bmask &= kv_map_block_mask(p, s, lb, lo, hi, lane);
                if (!bmask) continue;  // no run reaches into this block
              }
              for (int c0 = (r0 / p.rows) * p.rows; c0 < r1; c0 += p.rows) {
                // consumers read only the stage's rows, so a whole-block stage
                // carries the block mask as it is
                uint32_t cmask = bmask;
                if (p.rows < p.bs) {
                  cmask &= row_bits(c0, c0 + p.rows);
                  if (!cmask) continue;
                }
                if (p.pair) {
                  // hold the first block of a pair; emit both with the second
                  if (pend < 0) {
                    pend = phys;
                    pend_mask = cmask;
                    continue;
                  }
                  if (!emit(F_DATA | (first ? F_NEW : 0), s, 0, 2 * p.bs, pend, 0,
                            pend_mask | (cmask << 16), phys)) {
                    alive = false;
                    break;
                  }
                  pend = -1;
                  first = false;
                  continue;
                }
                if (!emit(F_DATA | (first ? F_NEW : 0), s, max(r0, c0), min(r1, c0 + p.rows),
                          phys, c0, cmask)) {
                  alive = false;
                  break;
                }
                first = false;
              }
              if (!alive) break;
            }
          }
          if (alive && pend >= 0) {
            // the segment's last block without a partner
            if (!emit(F_DATA | (first ? F_NEW : 0), s, 0, p.bs, pend, 0, pend_mask))
              alive = false;
            pend = -1;
            first = false;
          }
          if (alive && !emit(F_END | (first ? F_NEW : 0), s, 0, 0, -1, 0, 0u)) alive = false;
          x = seg_hi;
        }
        start += nb;
      }
    }
    if (alive) alive = emit(F_EXIT, 0, 0, 0, -1, 0, 0u);
    if (!alive) {
      // Stop: flag the others, then let every copy already issued land in
      // shared memory before this warp (and so the CTA) can retire.
      if (lane == 0) {
        *abort_flag = 1;
        report(p.status, MT_STATUS_BIT_TIMEOUT);
        const uint32_t first_live = it > (uint32_t)S ? it - (uint32_t)S : 0;
        for (uint32_t k = first_live; k < it; ++k) {
          const int slot = (int)(k % (uint32_t)S);
          volatile int never = 0;
          mbar_wait_bounded(&full[slot], (k / (uint32_t)S) & 1u, &never, p.wait_ns);
        }
      }
      __syncwarp();
    }
    return;
  }

  if (warp >= p.n_cw) return;
  pdl_wait();
  if (p.k_new) {
    // Appended rows outside every window are read by no CTA: the consumer
    // warps of CTA s mod grid write them while the first stages load. The
    // others are written by the producer of the CTA whose range loads their
    // block, just before it issues that block's copy.
    for (int s = blockIdx.x; s < p.B; s += gridDim.x) {
      const int lb = append_block(p, s);
      if (lb < 0) continue;
      int lo, hi;
      const int nb = seq_window(p, s, lo, hi);
      if (nb > 0 && lb >= lo / p.bs && lb < lo / p.bs + nb) continue;
      const int phys = p.table[(size_t)s * p.max_blocks + lb];
      if (phys < 0 || (long long)phys >= p.n_phys) {
        if (warp == 0 && lane == 0) report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
        continue;
      }
      append_row_part<FMT, D>(p, s, (long long)phys * p.bs + (p.ctx[s] - 1) % p.bs, lane, warp,
                              p.n_cw);
    }
  }
  if constexpr (MMA && FMT == MT_KV_Q8_0 && D == 128) {
    if (p.rows == 32)
      consume_q8_direct<GP, 2>(p, full, empty, infos, abort_flag, ring, scratch, warp, lane);
    else
      consume_q8_direct<GP, 1>(p, full, empty, infos, abort_flag, ring, scratch, warp, lane);
  } else if constexpr (MMA && FMT == MT_KV_Q8_0 && D <= 128) {
    consume_mma_q8<D, GP>(p, full, empty, infos, abort_flag, ring, smem + kHdrBytes, warp, lane);
  } else if constexpr (MMA) {
    consume_mma<FMT, D, GP>(p, full, empty, infos, abort_flag, ring, warp, lane);
  } else {
  // ------------------------------------------------------- consumer warps
  const int kvh = warp / p.wph;
  const int sub = warp % p.wph;
  const int tq = lane / C::LPT;           // token within a step
  const int j = lane % C::LPT;            // slice within the token
  const int hidx = j / C::REP;            // group head whose score this lane ends with
  const bool rep0 = (j % C::REP) == 0;
  const int rot = (C::LPT == 4 && C::NCL > 1) ? (tq & 1) : 0;  // bank-conflict rotation
  float *p_s = scratch + warp * scratch_floats_per_warp<GP>();
  float *a_s = p_s + 32 * GP;
  const int nsteps = p.bs / C::TPS;
  const int G = p.G;

  float qr[GP][C::DPL];
  float o_acc[GP][C::DV];
  float m_run = -INFINITY, l_run = 0.f;

  // element offset (within the head) of this lane's chunk k
  auto chunk_elem = [&](int k) -> int {
    if constexpr (FMT == MT_KV_Q8_0) {
      return C::DPL * j;
    } else {
      return (j + C::LPT * ((k + rot) % C::NCL)) * C::CH;
    }
  };

  for (RingPos rp;; rp.next(S)) {
    const int slot = (int)rp.slot;
    int okv = 1;
    if (lane == 0)
      okv = mbar_wait_bounded(&full[slot], rp.phase, abort_flag, p.wait_ns) ? 1 : 0;
    okv = __shfl_sync(kFull, okv, 0);
    if (!okv) {
      if (lane == 0) {
        *abort_flag = 1;
        report(p.status, MT_STATUS_BIT_TIMEOUT);
      }
      break;
    }
    struct {
      int seq, r0, r1, flags, base;
      uint32_t mask;
    } inf;
    {
      const volatile int *vi = reinterpret_cast<const volatile int *>(&infos[slot]);
      inf.seq = vi[0];
      inf.r0 = vi[1];
      inf.r1 = vi[2];
      inf.flags = vi[3] & 0xff;
      inf.base = vi[3] >> 8;
      inf.mask = (uint32_t)vi[4];
    }
    if (inf.flags & F_EXIT) break;
    const int seq = inf.seq;

    if (inf.flags & F_NEW) {
      const float *qb = p.q + ((size_t)seq * p.Hq + (size_t)kvh * G) * D;
#pragma unroll
      for (int g = 0; g < GP; ++g) {
#pragma unroll
        for (int k = 0; k < C::NCL; ++k) {
          const int e0 = chunk_elem(k);
#pragma unroll
          for (int e = 0; e < C::CH; e += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (g < G) v = *reinterpret_cast<const float4 *>(qb + (size_t)g * D + e0 + e);
            qr[g][k * C::CH + e + 0] = v.x * p.qscale;
            qr[g][k * C::CH + e + 1] = v.y * p.qscale;
            qr[g][k * C::CH + e + 2] = v.z * p.qscale;
            qr[g][k * C::CH + e + 3] = v.w * p.qscale;
          }
        }
#pragma unroll
        for (int e = 0; e < C::DV; ++e) o_acc[g][e] = 0.f;
      }
      m_run = -INFINITY;
      l_run = 0.f;
    }

    if (inf.flags & F_DATA) {
      // stage rows start at block row inf.base; steps never straddle stages
      const uint8_t *kst = ring + (size_t)slot * 2 * p.blk_pad - (ptrdiff_t)inf.base * p.row_bytes;
      const uint8_t *vst = kst + p.blk_pad;
      const int r0 = inf.r0, r1 = inf.r1;
      // ---- scores: Q.K for this lane's slice, reduced across the token's lanes
      // Raw scores go to this warp's scratch row p_s[token][head]; each lane
      // later reads back only the entries it wrote itself.
      float mloc = -INFINITY;
#pragma unroll 1
      for (int st = sub; st < nsteps; st += p.wph) {
        const int t0 = st * C::TPS;
        const int tok = t0 + tq;
        if (t0 + C::TPS <= r0 || t0 >= r1) {  // whole step outside the window
          if (rep0) p_s[tok * GP + hidx] = -INFINITY;
          continue;
        }
        float acc[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) acc[g] = 0.f;
        if constexpr (FMT == MT_KV_Q8_0) {
          const uint8_t *rowp = kst + (size_t)tok * p.row_bytes + kvh * (D / 32) * 34;
          const int b = (C::DPL * j) >> 5, o = (C::DPL * j) & 31;
          const uint8_t *qa = rowp + b * 34 + 2 + o;
          const uintptr_t a = reinterpret_cast<uintptr_t>(qa);
          const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
          const int sh = (int)(a & 3) * 8;
          constexpr int NW = C::DPL / 4;
          uint32_t raw[NW + 1];
#pragma unroll
          for (int i2 = 0; i2 <= NW; ++i2) raw[i2] = w[i2];
          const float dsc = __half2float(*reinterpret_cast<const __half *>(rowp + b * 34));
#pragma unroll
          for (int i2 = 0; i2 < NW; ++i2) {
            const uint32_t u = __funnelshift_r(raw[i2], raw[i2 + 1], sh) ^ 0x80808080u;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float x = i8_to_f(u, k);
#pragma unroll
              for (int g = 0; g < GP; ++g) acc[g] = fmaf(qr[g][i2 * 4 + k], x, acc[g]);
            }
          }
#pragma unroll
          for (int g = 0; g < GP; ++g) acc[g] *= dsc;
        } else {
          const uint8_t *rowp = kst + (size_t)tok * p.row_bytes + (size_t)kvh * D * C::ES;
#pragma unroll
          for (int k = 0; k < C::NCL; ++k) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(rowp + chunk_elem(k) * C::ES);
            float x[C::CH];
            if constexpr (FMT == MT_KV_F32) {
              x[0] = __uint_as_float(raw.x);
              x[1] = __uint_as_float(raw.y);
              x[2] = __uint_as_float(raw.z);
              x[3] = __uint_as_float(raw.w);
            } else {
              float2 f;
              f = h2_to_f2(raw.x); x[0] = f.x; x[1] = f.y;
              f = h2_to_f2(raw.y); x[2] = f.x; x[3] = f.y;
              f = h2_to_f2(raw.z); x[4] = f.x; x[5] = f.y;
              f = h2_to_f2(raw.w); x[6] = f.x; x[7] = f.y;
            }
#pragma unroll
            for (int e = 0; e < C::CH; ++e)
#pragma unroll
              for (int g = 0; g < GP; ++g) acc[g] = fmaf(qr[g][k * C::CH + e], x[e], acc[g]);
          }
        }
        halve<GP, C::LPT / 2>(acc, j);
        const bool valid = ((inf.mask >> tok) & 1u) && hidx < G;
        const float sc = valid ? acc[0] : -INFINITY;
        if (rep0) p_s[tok * GP + hidx] = sc;
        mloc = fmaxf(mloc, sc);
      }
      // ---- online softmax (base 2); the group's heads share nothing but
      // each head's max is common to all lanes that hold that head
#pragma unroll
      for (int o = C::LPT; o < 32; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, o));
      const float m_new = fmaxf(m_run, mloc);
      const bool none = m_new == -INFINITY;
      const float alpha = none ? 1.f : exp2f(m_run - m_new);
      l_run *= alpha;
      if (rep0) {
#pragma unroll 1
        for (int st = sub; st < nsteps; st += p.wph) {
          float *ps = p_s + (st * C::TPS + tq) * GP + hidx;
          const float pr = none ? 0.f : exp2f(*ps - m_new);
          l_run += pr;
          *ps = pr;
        }
      }
      m_run = m_new;
      if (tq == 0 && rep0) a_s[hidx] = alpha;
      __syncwarp();
      // ---- P.V: lane owns dims [lane*DV, lane*DV + DV) of every group head
      float al[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) al[g] = a_s[g];
#pragma unroll
      for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int e = 0; e < C::DV; ++e) o_acc[g][e] *= al[g];
      for (int i = 0; i < C::MAXSTEPS; ++i) {
        const int st = sub + p.wph * i;
        if (st >= nsteps) break;
        const int ta = max(st * C::TPS, r0), tb = min(st * C::TPS + C::TPS, r1);
        for (int tok = ta; tok < tb; ++tok) {
          if (!((inf.mask >> tok) & 1u)) continue;  // between kv_map runs
          float pg[GP];
          if constexpr (GP == 1) {
            pg[0] = p_s[tok];
          } else if constexpr (GP == 2) {
            const float2 v2 = *reinterpret_cast<const float2 *>(p_s + tok * 2);
            pg[0] = v2.x;
            pg[1] = v2.y;
          } else {
#pragma unroll
            for (int g = 0; g < GP; g += 4) {
              const float4 v4 = *reinterpret_cast<const float4 *>(p_s + tok * GP + g);
              pg[g] = v4.x;
              pg[g + 1] = v4.y;
              pg[g + 2] = v4.z;
              pg[g + 3] = v4.w;
            }
          }
          float x[C::DV];
          if constexpr (FMT == MT_KV_Q8_0) {
            const uint8_t *rowp = vst + (size_t)tok * p.row_bytes + kvh * (D / 32) * 34;
            const int dim0 = lane * C::DV;
            const int b = dim0 >> 5, o = dim0 & 31;
            const uintptr_t a = reinterpret_cast<uintptr_t>(rowp + b * 34 + 2 + o);
            const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
            const int sh = (int)(a & 3) * 8;
            constexpr int NWV = C::DV >= 4 ? C::DV / 4 : 1;
            uint32_t raw[NWV + 1];
#pragma unroll
            for (int i2 = 0; i2 <= NWV; ++i2) raw[i2] = w[i2];
            const float dsc = __half2float(*reinterpret_cast<const __half *>(rowp + b * 34));
#pragma unroll
            for (int i2 = 0; i2 < NWV; ++i2) {
              const uint32_t u = __funnelshift_r(raw[i2], raw[i2 + 1], sh) ^ 0x80808080u;
#pragma unroll
              for (int k = 0; k < 4 && i2 * 4 + k < C::DV; ++k) x[i2 * 4 + k] = i8_to_f(u, k);
            }
#pragma unroll
            for (int g = 0; g < GP; ++g) pg[g] *= dsc;
          } else if constexpr (FMT == MT_KV_F32) {
            const float *vp = reinterpret_cast<const float *>(vst + (size_t)tok * p.row_bytes) +
                              (size_t)kvh * D + lane * C::DV;
            if constexpr (C::DV == 2) {
              const float2 v2 = *reinterpret_cast<const float2 *>(vp);
              x[0] = v2.x;
              x[1] = v2.y;
            } else {
#pragma unroll
              for (int e = 0; e < C::DV; e += 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(vp + e);
                x[e] = v4.x;
                x[e + 1] = v4.y;
                x[e + 2] = v4.z;
                x[e + 3] = v4.w;
              }
            }
          } else {
            const uint8_t *vp = vst + (size_t)tok * p.row_bytes + ((size_t)kvh * D + lane * C::DV) * 2;
            if constexpr (C::DV == 2) {
              const float2 f = h2_to_f2(*reinterpret_cast<const uint32_t *>(vp));
              x[0] = f.x;
              x[1] = f.y;
            } else if constexpr (C::DV == 4) {
              const uint2 r = *reinterpret_cast<const uint2 *>(vp);
              float2 f = h2_to_f2(r.x);
              x[0] = f.x; x[1] = f.y;
              f = h2_to_f2(r.y);
              x[2] = f.x; x[3] = f.y;
            } else {
              const uint4 r = *reinterpret_cast<const uint4 *>(vp);
              float2 f = h2_to_f2(r.x);
              x[0] = f.x; x[1] = f.y;
              f = h2_to_f2(r.y);
              x[2] = f.x; x[3] = f.y;
              f = h2_to_f2(r.z);
              x[4] = f.x; x[5] = f.y;
              f = h2_to_f2(r.w);
              x[6] = f.x; x[7] = f.y;
            }
          }
#pragma unroll
          for (int g = 0; g < GP; ++g)
#pragma unroll
            for (int e = 0; e < C::DV; ++e) o_acc[g][e] = fmaf(pg[g], x[e], o_acc[g][e]);
        }
      }
      __syncwarp();
    }

    if (inf.flags & F_END) {
      float lsum = l_run;  // non-zero only on the rep0 lanes
#pragma unroll
      for (int o = C::LPT; o < 32; o <<= 1) lsum += __shfl_xor_sync(kFull, lsum, o);
      const size_t P = ((size_t)blockIdx.x + seq) * p.n_sub + sub;
      const size_t hq0 = P * p.Hq + (size_t)kvh * G;
      if (tq == 0 && rep0 && hidx < G) {
        p.part_ml[(hq0 + hidx) * 2 + 0] = m_run;
        p.part_ml[(hq0 + hidx) * 2 + 1] = lsum;
      }
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        if (g >= G) break;
        float *dst = p.part_o + (hq0 + g) * D + lane * C::DV;
#pragma unroll
        for (int e = 0; e < C::DV; e += 2)
          *reinterpret_cast<float2 *>(dst + e) = make_float2(o_acc[g][e], o_acc[g][e + 1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  }  // SIMT consumers
}

// Merge every partial of (sequence, query head) by log-sum-exp and
// normalise. One warp per (s, h); lane owns D/32 output dims. The (m, l)
// pairs of up to 32 partials arrive in one round (a lane each); the output
// partials then stream in with several loads in flight; longer lists are
// taken 32 at a time with an online rescale.
template <int D>
__global__ void __launch_bounds__(256) splitk_combine_kernel(const Params p) {
  constexpr int DV = D / 32;
  pdl_trigger();
  // With few (s, h) pairs, wps warps share one pair's partial list (each a
  // contiguous share) and merge their results through shared memory.
  __shared__ float red_s[8][2 + D];
  const int wps = p.combine_wps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * (8 / wps) + warp / wps;
  const int kw = warp % wps;
  const bool live = w < p.B * p.Hq;
  const int s = live ? w / p.Hq : 0, h = live ? w % p.Hq : 0;
  // the sequence's first stream position and the stream length follow from
  // the context lengths and windows (read-only inputs, the decode's own
  // arithmetic), so they are computed before waiting for the decode
  int T = 0, beg = 0, end = 0;
  for (int base = 0; base < p.B; base += 32) {
    const int sl = base + lane;
    int lo, hi, nb = 0;
    if (sl < p.B) nb = seq_window(p, sl, lo, hi);
    const int incl = warp_incl_scan(nb, lane);
    if (s >= base && s < base + 32) {
      const int incl_s = __shfl_sync(kFull, incl, s - base);
      const int nb_s = __shfl_sync(kFull, nb, s - base);
      beg = T + incl_s - nb_s;
      end = T + incl_s;
    }
    T += __shfl_sync(kFull, incl, 31);
  }
  pdl_wait();
  const int per = T > 0 ? (T + p.n_ctas - 1) / p.n_ctas : 1;
  float acc[DV];
#pragma unroll
  for (int e = 0; e < DV; ++e) acc[e] = 0.f;
  float M = -INFINITY, L = 0.f;
  // The partials of (s, h): the decode's (CTA-major, n_sub per CTA), then,
  // for a sequence of a shared-prefix group, the prefix kernel's records of
  // its tile (one per prefix CTA whose range meets the tile).
  const int c0 = end > beg ? beg / per : 0;
  const int NPd = end > beg ? ((end - 1) / per - c0 + 1) * p.n_sub : 0;
  int NPc = 0, Tc = 0, Rc = 0, cc0 = 0;
  if (p.casc.n_groups) {
    long long u0 = 0;
    const int gi = cascade_find(p.casc, p.Hkv, p.G, s, h, Tc, Rc, u0);
    if (gi >= 0 && p.casc.g[gi].nblk > 0) {
      cc0 = (int)(u0 / p.casc.per);
      NPc = (int)((u0 + p.casc.g[gi].nblk - 1) / p.casc.per) - cc0 + 1;
    }
  }
  const int NP_all = live ? NPd + NPc : 0;
  const int i_beg = kw * NP_all / wps, i_end = (kw + 1) * NP_all / wps;
  const int NP = i_end - i_beg;
  auto part = [&](int i, const float *&ml, const float *&o) {
    i += i_beg;
    if (i < NPd) {
      const size_t P = ((size_t)c0 + i / p.n_sub + s) * p.n_sub + i % p.n_sub;
      ml = p.part_ml + (P * p.Hq + h) * 2;
      o = p.part_o + (P * p.Hq + h) * D;
    } else {
      const size_t slot = (size_t)cc0 + (i - NPd) + Tc;
      ml = p.casc.rec_ml + (slot * kPrefixRows + Rc) * 2;
      o = p.casc.rec_o + (slot * kPrefixRows + Rc) * D;
    }
  };
  // Per round of up to 32 partials: the (m, l) pairs (a lane each) and the
  // output rows of the first KB partials are all requested before any is
  // used, so a list of up to KB partials costs one L2 round trip. Every
  // listed partial was written by its kernel (zeros where it saw nothing),
  // so the loads need no validity test; weights of empty partials are 0.
  constexpr int KB = DV >= 8 ? 8 : 16;
  for (int base = 0; base < NP; base += 32) {
    const int cnt = min(32, NP - base);
    float m = -INFINITY, l = 0.f;
    if (lane < cnt) {
      const float *mlp, *op;
      part(base + lane, mlp, op);
      const float2 ml = *reinterpret_cast<const float2 *>(mlp);
      m = ml.x;
      l = ml.y;
    }
    float v[KB][DV];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      if (j < cnt) {
        const float *mlp, *op;
        part(base + j, mlp, op);
        const float *src = op + lane * DV;
        if constexpr (DV % 4 == 0) {
#pragma unroll
          for (int e = 0; e < DV; e += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src + e);
            v[j][e] = x.x;
            v[j][e + 1] = x.y;
            v[j][e + 2] = x.z;
            v[j][e + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < DV; e += 2) {
            const float2 x = *reinterpret_cast<const float2 *>(src + e);
            v[j][e] = x.x;
            v[j][e + 1] = x.y;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < DV; ++e) v[j][e] = 0.f;
      }
    }
    if (!(l > 0.f)) m = -INFINITY;
    float mc = m;
#pragma unroll
    for (int o = 16; o; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kFull, mc, o));
    const float m_new = fmaxf(M, mc);
    if (m_new == -INFINITY) continue;  // nothing valid yet
    const float f_old = exp2f(M - m_new);
    const float f = m == -INFINITY ? 0.f : exp2f(m - m_new);
    float lc = l * f;
#pragma unroll
    for (int o = 16; o; o >>= 1) lc += __shfl_xor_sync(kFull, lc, o);
    L = L * f_old + lc;
    M = m_new;
#pragma unroll
    for (int e = 0; e < DV; ++e) acc[e] *= f_old;
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      const float fk = __shfl_sync(kFull, f, j);
#pragma unroll
      for (int e = 0; e < DV; ++e) acc[e] = fmaf(fk, v[j][e], acc[e]);
    }
    // partials beyond the first KB of the round, KB at a time
    for (int k0 = KB; k0 < cnt; k0 += KB) {
      float fk[KB];
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        fk[j] = __shfl_sync(kFull, f, (k0 + j) & 31);
        if (k0 + j < cnt) {
          const float *mlp, *op;
          part(base + k0 + j, mlp, op);
          const float *src = op + lane * DV;
#pragma unroll
          for (int e = 0; e < DV; e += 2) {
            const float2 x = *reinterpret_cast<const float2 *>(src + e);
            v[j][e] = x.x;
            v[j][e + 1] = x.y;
          }
        } else {
          fk[j] = 0.f;
#pragma unroll
          for (int e = 0; e < DV; ++e) v[j][e] = 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < KB; ++j)
#pragma unroll
        for (int e = 0; e < DV; ++e) acc[e] = fmaf(fk[j], v[j][e], acc[e]);
    }
  }
  if (wps > 1) {
    if (lane == 0) {
      red_s[warp][0] = M;
      red_s[warp][1] = L;
    }
#pragma unroll
    for (int e = 0; e < DV; ++e) red_s[warp][2 + lane * DV + e] = acc[e];
    __syncthreads();
    if (kw == 0) {
      float Mx = -INFINITY;
      for (int i = 0; i < wps; ++i)
        if (red_s[warp + i][1] > 0.f) Mx = fmaxf(Mx, red_s[warp + i][0]);
      L = 0.f;
#pragma unroll
      for (int e = 0; e < DV; ++e) acc[e] = 0.f;
      if (Mx != -INFINITY) {
        for (int i = 0; i < wps; ++i) {
          const float li = red_s[warp + i][1];
          if (!(li > 0.f)) continue;
          const float f = exp2f(red_s[warp + i][0] - Mx);
          L = fmaf(f, li, L);
#pragma unroll
          for (int e = 0; e < DV; ++e) acc[e] = fmaf(f, red_s[warp + i][2 + lane * DV + e], acc[e]);
        }
      }
      M = Mx;
    }
  }
  if (!live || kw != 0) return;
  float *dst = p.out + ((size_t)s * p.Hq + h) * D + lane * DV;
  const bool any = L > 0.f;
  const float inv = any ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < DV; e += 2)
    *reinterpret_cast<float2 *>(dst + e) = make_float2(acc[e] * inv, acc[e + 1] * inv);
  if (p.lse && lane == 0)
    p.lse[(size_t)s * p.Hq + h] = any ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
}

// --------------------------------------------------------------- host side

struct Plan {
  int D, GP, wph, n_cw, stages, n_ctas, blk_pad, rows, smem;
  bool mma;
  int pitch, n_sub, ncb, scratch;
  int q8_chunk;  // q8_0 staged through the word tensor map: chunk bytes (0: bulk copies)
  bool two_per_sm;  // kernel compiled for two resident CTAs per SM
  bool pair;        // q8_0 block size 16: two blocks per 32-row stage
  size_t ws_status, ws_ml, ws_o, ws_total;
};

int pad_group(int G) {
  if (G <= 1) return 1;
  if (G <= 2) return 2;
  if (G <= 4) return 4;
  if (G <= 8) return 8;
  return 0;
}

mt_status make_plan(const mt_paged_attn_args *a, Plan *pl, bool need_device) {
  if (!a) return fail(MT_ERR_INVALID_ARG, "paged decode: null args");
  const size_t rb = mt_kv_row_bytes(a->fmt, a->n_kv_heads, a->head_dim);
  if (rb == 0) return fail(MT_ERR_INVALID_ARG, "paged decode: unknown format or bad head shape");
  if (a->n_seqs < 0 || a->n_heads <= 0 || a->max_blocks < 0 || a->n_phys_blocks < 0 ||
      a->block_size <= 0)
    return fail(MT_ERR_INVALID_ARG, "paged decode: negative or zero size");
  if (a->n_heads % a->n_kv_heads)
    return fail(MT_ERR_INVALID_ARG, "paged decode: n_heads must be a multiple of n_kv_heads");
  if (a->spans && a->kv_map)
    return fail(MT_ERR_INVALID_ARG,
                "paged decode: spans and kv_map are two window modes: pass at most one");
  if (a->head_dim != 64 && a->head_dim != 128 && a->head_dim != 256)
    return fail(MT_ERR_UNSUPPORTED, "paged decode: head_dim must be 64, 128 or 256");
  if (a->block_size != 16 && a->block_size != 32)
    return fail(MT_ERR_UNSUPPORTED, "paged decode: block_size must be 16 or 32");
  if (a->n_kv_heads > kMaxConsumerWarps)
    return fail(MT_ERR_UNSUPPORTED, "paged decode: at most 8 KV heads");
  const int G = a->n_heads / a->n_kv_heads;
  const int GP = pad_group(G);
  if (!GP) return fail(MT_ERR_UNSUPPORTED, "paged decode: at most 8 query heads per KV head");
  if (a->n_ctas < 0) return fail(MT_ERR_INVALID_ARG, "paged decode: negative n_ctas");
  if ((long long)a->max_blocks * a->block_size > 0x7fffffffLL)
    return fail(MT_ERR_UNSUPPORTED, "paged decode: max_blocks * block_size overflows int32");
  pl->D = a->head_dim;
  pl->GP = GP;
  // header, scratch (softmax rows, or the q8_0 conversion tiles), 1024 bytes
  // to align the ring, 16 bytes of tail
  const bool q8_mma = a->fmt == MT_KV_Q8_0 && (a->head_dim == 64 || a->head_dim == 128);
  const int simt_scratch = (kMaxConsumerWarps * (32 * GP + GP) * 4 + 127) & ~127;
  // (per warp: K and V tiles of 16 rows, then their f32 group scales; for
  // head_dim 128 the operands come straight from the staged rows and only
  // the f32 scale arrays are kept)
  const bool q8_direct = q8_mma && a->head_dim == 128;
  const int tile_scratch =
      q8_direct ? kMaxConsumerWarps * 2 * kQ8dScaleFloatsPerHalf * 4
                : kMaxConsumerWarps * 2 * 16 * ((2 * a->head_dim + 16) + (a->head_dim / 32) * 4);
  // (the direct q8_0 consumer uses only its scale arrays)
  pl->scratch = q8_direct ? tile_scratch
                          : (q8_mma ? std::max(simt_scratch, tile_scratch) : simt_scratch);
  int fixed = kHdrBytes + pl->scratch + 1024 + 16;
  int n_ctas = a->n_ctas;
  const bool auto_ctas = n_ctas == 0;
  int smem_cap = 232448;
  if (need_device || n_ctas == 0) {
    DeviceInfo di;
    mt_status st = device_info(&di);
    if (st != MT_OK) return st;
    if (n_ctas == 0) n_ctas = di.n_sm;
    smem_cap = di.smem_optin;
  }
  // Rows per stage: whole blocks when at least two stages fit, else halve
  // (never below `min_rows`). Returns false when even that does not fit.
  auto fit = [&](int pitch, int min_rows, int &rows, int &pad, int &stages) {
    rows = a->block_size;
    for (;;) {
      pad = (int)(((size_t)rows * pitch + 127) & ~(size_t)127);
      stages = (smem_cap - fixed) / (2 * pad);
      if (stages >= 2 || rows <= min_rows) break;
      rows /= 2;
    }
    if (stages > kMaxStages) stages = kMaxStages;
    return stages >= 2 && rows >= min_rows;
  };
  int rows = 0, pad = 0, stages = 0, wph = 1;
  // f16 and f32 pools use the tensor-core consumers when a warp per KV head
  // (two for head_dim 256) fits in the 8 consumer warps and 16-row stages fit.
  const int mma_wph = a->head_dim == 256 ? 2 : 1;
  const int nc = (int)(rb / 128);
  pl->ncb = nc | 1;  // odd number of 128-byte lines per staged row
  // (f32 pools: head_dim 64 and 128; at 256 the split operands do not fit in
  // registers and those pools stay on the FP32-core consumers)
  // (f32 pools whose 16-row stages do not fit twice take 8-row stages)
  pl->mma = (a->fmt == MT_KV_F16 || (a->fmt == MT_KV_F32 && a->head_dim <= 128)) &&
            rb % 128 == 0 && pl->ncb <= 255 &&
            a->n_kv_heads * mma_wph <= kMaxConsumerWarps &&
            fit(128 * pl->ncb, a->fmt == MT_KV_F32 ? 8 : 16, rows, pad, stages);
  // q8_0 pools: tensor-core consumers (d <= 128). For head_dim 128 the rows
  // are staged by a tensor copy whose box is wider than the row when the
  // row is whole 32- or 16-byte chunks, so that the staged pitch is 8 or 24
  // banks mod 32 (rows 4 apart share a bank group, rows 1 to 3 apart do
  // not): the consumer's per-token loads then hit distinct banks.
  pl->q8_chunk = 0;
  int q8_pitch = (int)rb;
  if (!pl->mma && q8_mma && a->head_dim == 128) {
    if (rb % 32 == 0) {
      const int nch = (int)(rb / 32);
      q8_pitch = 32 * (nch | 1);
      pl->q8_chunk = 32;
    } else if (rb % 16 == 0) {
      int nch = (int)(rb / 16);
      while (nch % 4 != 2) ++nch;
      q8_pitch = 16 * nch;
      pl->q8_chunk = 16;
    }
    if (pl->q8_chunk && q8_pitch / pl->q8_chunk > 256) {  // a box dimension holds at most 256
      pl->q8_chunk = 0;
      q8_pitch = (int)rb;
    }
  }
  // At block size 16 the direct consumer takes two blocks of a sequence per
  // 32-row stage (one tensor copy each), so that each warp works on two
  // independent 16-row halves per stage as at block size 32.
  pl->pair = false;
  if (!pl->mma && q8_mma && pl->q8_chunk && a->block_size == 16) {
    const int pad2 = (32 * q8_pitch + 127) & ~127;
    const int st2 = std::min((smem_cap - fixed) / (2 * pad2), kMaxStages);
    if (st2 >= 2) {
      pl->pair = true;
      pl->mma = true;
      wph = 1;
      pl->pitch = q8_pitch;
      pl->n_sub = 1;
      rows = 32;
      pad = pad2;
      stages = st2;
    }
  }
  if (pl->pair) {
  } else if (!pl->mma && q8_mma && fit(q8_pitch, 16, rows, pad, stages)) {
    pl->mma = true;
    wph = 1;
    pl->pitch = q8_pitch;
    pl->n_sub = 1;
  } else if (pl->mma) {
    wph = mma_wph;
    pl->pitch = 128 * pl->ncb;
    pl->n_sub = 1;
  } else {
    const int dpl = GP >= 8 ? 8 : 16;
    const int tps = 32 / (a->head_dim / dpl);
    const int nsteps = a->block_size / tps;
    wph = kMaxConsumerWarps / a->n_kv_heads;
    if (wph > nsteps) wph = nsteps;
    if (wph < 1) wph = 1;
    // the FP32-core consumers keep their softmax rows in the scratch
    pl->scratch = std::max(pl->scratch, simt_scratch);
    fixed = kHdrBytes + pl->scratch + 1024 + 16;
    if (!fit((int)rb, 8, rows, pad, stages))
      return fail(MT_ERR_UNSUPPORTED, "paged decode: KV rows too wide to double-buffer 8 of them");
    pl->pitch = (int)rb;
    pl->n_sub = wph;
  }
  pl->wph = wph;
  pl->n_cw = a->n_kv_heads * wph;
  // Few consumer warps (pools with few KV heads, narrow rows): two CTAs per
  // SM, each with stages sized for half of the SM's shared memory, so every
  // scheduler runs two consumer warps. With at most 4 warps per CTA (one per
  // scheduler) two CTAs always fit the per-scheduler register file.
  // The direct q8_0 consumer at block size 16 without paired stages (rows
  // that are not whole 16-byte chunks) also runs two CTAs per SM: 16-row
  // stages, and a kernel compiled for two resident CTAs when a CTA has more
  // than 3 consumer warps. Paired stages keep their 32 rows and their
  // two-half scale arrays.
  pl->two_per_sm = false;
  if (auto_ctas && (pl->n_cw <= 3 || (q8_direct && pl->mma && !pl->pair && a->block_size == 16))) {
    const int min_rows = pl->mma ? 16 : 8;
    int rows2 = 0, pad2 = 0, stages2 = 0;
    const int cap1 = smem_cap, fixed1 = fixed, scratch1 = pl->scratch;
    smem_cap = (cap1 + 1024) / 2 - 1024;
    bool fits;
    if (pl->pair) {
      rows2 = 32;
      pad2 = (32 * pl->pitch + 127) & ~127;
      stages2 = std::min((smem_cap - fixed) / (2 * pad2), kMaxStages);
      fits = true;
    } else if (q8_direct && pl->mma) {
      // 16-row stages: scale arrays for one half
      pl->scratch = kMaxConsumerWarps * kQ8dScaleFloatsPerHalf * 4;
      fixed = kHdrBytes + pl->scratch + 1024 + 16;
      fits = fit(pl->pitch, min_rows, rows2, pad2, stages2) && rows2 == 16;
    } else {
      fits = fit(pl->pitch, min_rows, rows2, pad2, stages2);
    }
    if (fits && stages2 >= 3) {
      rows = rows2;
      pad = pad2;
      stages = stages2;
      n_ctas *= 2;
      pl->two_per_sm = q8_direct && pl->mma && pl->n_cw > 3;
    } else {
      fixed = fixed1;
      pl->scratch = scratch1;
    }
    smem_cap = cap1;
  }
  pl->rows = rows;
  pl->blk_pad = pad;
  pl->stages = stages;
  pl->smem = fixed + stages * 2 * pl->blk_pad;
  pl->n_ctas = n_ctas;
  const size_t P = ((size_t)n_ctas + (size_t)a->n_seqs) * pl->n_sub;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  pl->ws_status = 0;
  pl->ws_ml = 256;
  pl->ws_o = pl->ws_ml + up(P * a->n_heads * 2 * 4);
  pl->ws_total = pl->ws_o + up(P * a->n_heads * (size_t)a->head_dim * 4);
  return MT_OK;
}

template <int FMT, int D, int GP, bool MMA, int MINB>
mt_status launch_decode_k(const Params &prm, const Plan &pl, cudaStream_t s) {
  auto kern = paged_decode_kernel<FMT, D, GP, MMA, MINB>;
  mt_status st = kernel_smem(reinterpret_cast<const void *>(kern), pl.smem,
                             "cudaFuncSetAttribute(decode smem)", true);
  if (st != MT_OK) return st;
  st = cuda_check(
      launch_pdl(kern, dim3(pl.n_ctas), dim3(32 * (pl.n_cw + 1)), pl.smem, s, prm),
      "paged decode launch");
  if (st != MT_OK) return st;
  const int warps = prm.B * prm.Hq * prm.combine_wps;
  if (warps > 0) {
    st = cuda_check(launch_pdl(splitk_combine_kernel<D>, dim3((warps + 7) / 8), dim3(256), 0, s,
                               prm),
                    "split-K combine launch");
  }
  return st;
}

template <int FMT, int D, int GP, bool MMA>
mt_status launch_decode(const Params &prm, const Plan &pl, cudaStream_t s) {
  if constexpr (MMA && FMT == MT_KV_Q8_0 && D == 128) {
    if (pl.two_per_sm) return launch_decode_k<FMT, D, GP, MMA, 2>(prm, pl, s);
  }
  return launch_decode_k<FMT, D, GP, MMA, 1>(prm, pl, s);
}

template <int FMT, int D, bool MMA>
mt_status dispatch_gp(const Params &prm, const Plan &pl, cudaStream_t s) {
  switch (pl.GP) {
    case 1: return launch_decode<FMT, D, 1, MMA>(prm, pl, s);
    case 2: return launch_decode<FMT, D, 2, MMA>(prm, pl, s);
    case 4: return launch_decode<FMT, D, 4, MMA>(prm, pl, s);
    default: return launch_decode<FMT, D, 8, MMA>(prm, pl, s);
  }
}

template <int FMT, bool MMA>
mt_status dispatch_d(const Params &prm, const Plan &pl, cudaStream_t s) {
  switch (pl.D) {
    case 64: return dispatch_gp<FMT, 64, MMA>(prm, pl, s);
    case 128: return dispatch_gp<FMT, 128, MMA>(prm, pl, s);
    // f32 pools of head_dim 256 always take the FP32-core consumers (plan)
    default: return dispatch_gp<FMT, 256, MMA && FMT != MT_KV_F32>(prm, pl, s);
  }
}

// 3-D tensor map of a pool for the tensor-core path: [cells][row chunks of
// 128 bytes][64 f16], box = (64, ncb, rows), 128-byte swizzle, zero fill.
// q8_0 pools (head_dim 128): [cells][row chunks][32-bit words], box =
// (chunk words, pitch / chunk, rows), no swizzle, zero fill.
mt_status encode_pool_map(CUtensorMap *map, const void *pool, long long n_cells, size_t rb,
                          const Plan &pl) {
  if (pl.q8_chunk)
    return encode_pool_map_words(map, pool, n_cells, rb, pl.q8_chunk, pl.pitch / pl.q8_chunk,
                                 pl.pair ? pl.rows / 2 : pl.rows);
  return encode_pool_map_3d(map, pool, n_cells, rb, pl.ncb, pl.rows);
}

// Fill the kernel parameters shared by both decode entry points.
mt_status fill_params(Params &prm, const mt_paged_attn_args *a, const Plan &pl, uint8_t *ws,
                      uint32_t *status) {
  prm.q = a->q;
  prm.k_pool = static_cast<const uint8_t *>(a->k_pool);
  prm.v_pool = static_cast<const uint8_t *>(a->v_pool);
  prm.table = a->block_table;
  prm.ctx = a->context_lens;
  prm.spans = a->spans;
  prm.kv_map = a->kv_map;
  prm.out = a->out;
  prm.lse = a->lse;
  prm.status = status;
  prm.k_new = nullptr;
  prm.v_new = nullptr;
  prm.casc.n_groups = 0;
  prm.part_ml = reinterpret_cast<float *>(ws + pl.ws_ml);
  prm.part_o = reinterpret_cast<float *>(ws + pl.ws_o);
  prm.B = a->n_seqs;
  prm.Hq = a->n_heads;
  prm.Hkv = a->n_kv_heads;
  prm.G = a->n_heads / a->n_kv_heads;
  prm.bs = a->block_size;
  prm.max_blocks = a->max_blocks;
  prm.n_phys = a->n_phys_blocks;
  prm.row_bytes = (int)mt_kv_row_bytes(a->fmt, a->n_kv_heads, a->head_dim);
  prm.blk_pad = pl.blk_pad;
  prm.rows = pl.rows;
  prm.pitch = pl.pitch;
  prm.use_tmap = (pl.mma && (a->fmt == MT_KV_F16 || a->fmt == MT_KV_F32 || pl.q8_chunk)) ? 1 : 0;
  prm.pair = pl.pair ? 1 : 0;
  prm.scratch_bytes = pl.scratch;
  prm.ncb = pl.ncb;
  prm.n_sub = pl.n_sub;
  prm.stages = pl.stages;
  prm.wph = pl.wph;
  prm.n_cw = pl.n_cw;
  prm.n_ctas = pl.n_ctas;
  prm.qscale = a->scale * 1.4426950408889634f;
  prm.wait_ns = kWaitLimitNs;
  // about 2048 combine warps: small batches split each pair's partial list
  {
    const long long pairs = (long long)a->n_seqs * a->n_heads;
    int wps = 1;
    while (wps < 8 && pairs * wps < 2048) wps *= 2;
    prm.combine_wps = wps;
  }
  if (prm.use_tmap) {
    const long long n_cells = (long long)a->n_phys_blocks * a->block_size;
    const size_t rb = (size_t)prm.row_bytes;
    mt_status st = encode_pool_map(&prm.tmap_k, a->k_pool, n_cells, rb, pl);
    if (st != MT_OK) return st;
    st = encode_pool_map(&prm.tmap_v, a->v_pool, n_cells, rb, pl);
    if (st != MT_OK) return st;
  }
  return MT_OK;
}

mt_status dispatch(const Params &prm, const Plan &pl, mt_kv_format fmt, cudaStream_t s) {
  switch (fmt) {
    case MT_KV_F32:
      return pl.mma ? dispatch_d<MT_KV_F32, true>(prm, pl, s)
                    : dispatch_d<MT_KV_F32, false>(prm, pl, s);
    case MT_KV_F16:
      return pl.mma ? dispatch_d<MT_KV_F16, true>(prm, pl, s)
                    : dispatch_d<MT_KV_F16, false>(prm, pl, s);
    default:
      return pl.mma ? dispatch_d<MT_KV_Q8_0, true>(prm, pl, s)
                    : dispatch_d<MT_KV_Q8_0, false>(prm, pl, s);
  }
}

}  // namespace
}  // namespace mtkv

using namespace mtkv;

extern "C" size_t mt_paged_attn_workspace_bytes(const mt_paged_attn_args *args) {
  Plan pl;
  if (make_plan(args, &pl, false) != MT_OK) return 0;
  return pl.ws_total;
}

extern "C" mt_status mt_paged_attn_decode(const mt_paged_attn_args *a, void *workspace,
                                          size_t workspace_bytes, mt_stream stream) {
  Plan pl;
  mt_status st = make_plan(a, &pl, true);
  if (st != MT_OK) return st;
  if (a->n_seqs == 0) return ok();
  if (!a->q || !a->k_pool || !a->v_pool || !a->block_table || !a->context_lens || !a->out)
    return fail(MT_ERR_INVALID_ARG, "paged decode: null pointer");
  if (!workspace || workspace_bytes < pl.ws_total)
    return fail(MT_ERR_INVALID_ARG, "paged decode: workspace missing or too small (need " +
                                        std::to_string(pl.ws_total) + " bytes)");
  if (!aligned16(a->k_pool) || !aligned16(a->v_pool) || !aligned16(a->q) || !aligned16(a->out) ||
      !aligned16(workspace))
    return fail(MT_ERR_INVALID_ARG, "paged decode: q, pools, out and workspace must be 16-byte aligned");
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  Params prm;
  st = fill_params(prm, a, pl, ws, reinterpret_cast<uint32_t *>(ws + pl.ws_status));
  if (st != MT_OK) return st;
  st = dispatch(prm, pl, a->fmt, reinterpret_cast<cudaStream_t>(stream));
  return st == MT_OK ? ok() : st;
}

// ------------------------------------------------- shared-prefix (cascade)

namespace mtkv {
namespace {

struct CascadePlan {
  bool use;          // the prefix kernel covers the shape (else: plain decode)
  Cascade c;
  size_t rec_off;    // records start (bytes into the workspace)
  size_t total;      // workspace bytes
};

mt_status cascade_plan(const mt_paged_attn_args *a, const Plan &pl,
                       const mt_prefix_group *groups, int n_groups, CascadePlan *cp) {
  if (n_groups < 0) return fail(MT_ERR_INVALID_ARG, "cascade decode: negative group count");
  if (n_groups > kMaxPrefixGroups)
    return fail(MT_ERR_UNSUPPORTED, "cascade decode: at most 64 prefix groups");
  if (n_groups > 0 && !groups) return fail(MT_ERR_INVALID_ARG, "cascade decode: null groups");
  std::vector<std::pair<int, int>> spans;
  for (int i = 0; i < n_groups; ++i) {
    const mt_prefix_group &g = groups[i];
    if (g.seq_begin < 0 || g.seq_end > a->n_seqs || g.seq_begin >= g.seq_end)
      return fail(MT_ERR_INVALID_ARG, "cascade decode: group " + std::to_string(i) +
                                          " has an empty or out-of-range sequence range");
    if (g.n_prefix_blocks < 0 || g.n_prefix_blocks > a->max_blocks)
      return fail(MT_ERR_INVALID_ARG,
                  "cascade decode: group " + std::to_string(i) + " prefix outside the table");
    spans.emplace_back(g.seq_begin, g.seq_end);
  }
  std::sort(spans.begin(), spans.end());
  for (size_t i = 1; i < spans.size(); ++i)
    if (spans[i].first < spans[i - 1].second)
      return fail(MT_ERR_INVALID_ARG, "cascade decode: prefix groups overlap");
  cp->total = pl.ws_total;
  cp->rec_off = pl.ws_total;
  Cascade &c = cp->c;
  c = Cascade{};
  cp->use = n_groups > 0 && prefix_supported(a->fmt, a->head_dim, a->block_size, pl.GP);
  if (!cp->use) return MT_OK;
  c.n_groups = n_groups;
  c.gp = pl.GP;
  c.tq = kPrefixRows / pl.GP;
  long long tiles = 0, units = 0;
  for (int i = 0; i < n_groups; ++i) {
    c.g[i] = PrefixGroup{groups[i].seq_begin, groups[i].seq_end, groups[i].n_prefix_blocks};
    const long long t = (long long)cascade_qtiles(c, i) * a->n_kv_heads;
    tiles += t;
    units += t * groups[i].n_prefix_blocks;
  }
  DeviceInfo di;
  mt_status st = device_info(&di);
  if (st != MT_OK) return st;
  const long long ctas =
      std::min<long long>((long long)di.n_sm * prefix_ctas_per_sm(a->head_dim), units);
  c.n_tiles = (int)tiles;
  c.n_units = units;
  c.n_ctas = ctas > 0 ? (int)ctas : 0;
  c.per = ctas > 0 ? (int)((units + ctas - 1) / ctas) : 1;
  const size_t slots = (size_t)c.n_ctas + (size_t)c.n_tiles;
  const size_t ml_bytes = (slots * kPrefixRows * 2 * 4 + 255) & ~(size_t)255;
  const size_t o_bytes = slots * kPrefixRows * (size_t)a->head_dim * 4;
  cp->total = cp->rec_off + ml_bytes + o_bytes;
  return MT_OK;
}

}  // namespace
}  // namespace mtkv

extern "C" size_t mt_paged_attn_cascade_workspace_bytes(const mt_paged_attn_args *a,
                                                        const mt_prefix_group *groups,
                                                        int n_groups) {
  Plan pl;
  if (make_plan(a, &pl, false) != MT_OK) return 0;
  CascadePlan cp;
  if (cascade_plan(a, pl, groups, n_groups, &cp) != MT_OK) return 0;
  return cp.total;
}

namespace mtkv {
namespace {
mt_status cascade_decode(const mt_paged_attn_args *a, const mt_prefix_group *groups, int n_groups,
                         const float *k_new, const float *v_new, void *workspace,
                         size_t workspace_bytes, mt_stream stream);
}  // namespace
}  // namespace mtkv

extern "C" mt_status mt_paged_attn_decode_cascade(const mt_paged_attn_args *a,
                                                  const mt_prefix_group *groups, int n_groups,
                                                  void *workspace, size_t workspace_bytes,
                                                  mt_stream stream) {
  return cascade_decode(a, groups, n_groups, nullptr, nullptr, workspace, workspace_bytes, stream);
}

extern "C" mt_status mt_paged_attn_decode_cascade_append(const mt_paged_attn_args *a,
                                                         const mt_prefix_group *groups,
                                                         int n_groups, const float *k_new,
                                                         const float *v_new, void *workspace,
                                                         size_t workspace_bytes,
                                                         mt_stream stream) {
  if (!k_new || !v_new)
    return fail(MT_ERR_INVALID_ARG, "cascade decode with append: null new rows");
  return cascade_decode(a, groups, n_groups, k_new, v_new, workspace, workspace_bytes, stream);
}

namespace mtkv {
namespace {
mt_status cascade_decode(const mt_paged_attn_args *a, const mt_prefix_group *groups, int n_groups,
                         const float *k_new, const float *v_new, void *workspace,
                         size_t workspace_bytes, mt_stream stream) {
  Plan pl;
  mt_status st = make_plan(a, &pl, true);
  if (st != MT_OK) return st;
  CascadePlan cp;
  st = cascade_plan(a, pl, groups, n_groups, &cp);
  if (st != MT_OK) return st;
  if (a->n_seqs == 0) return ok();
  if (!a->q || !a->k_pool || !a->v_pool || !a->block_table || !a->context_lens || !a->out)
    return fail(MT_ERR_INVALID_ARG, "cascade decode: null pointer");
  if (!workspace || workspace_bytes < cp.total)
    return fail(MT_ERR_INVALID_ARG, "cascade decode: workspace missing or too small (need " +
                                        std::to_string(cp.total) + " bytes)");
  if (!aligned16(a->k_pool) || !aligned16(a->v_pool) || !aligned16(a->q) || !aligned16(a->out) ||
      !aligned16(workspace))
    return fail(MT_ERR_INVALID_ARG,
                "cascade decode: q, pools, out and workspace must be 16-byte aligned");
  if ((k_new && !aligned16(k_new)) || (v_new && !aligned16(v_new)))
    return fail(MT_ERR_INVALID_ARG, "cascade decode with append: new rows must be 16-byte aligned");
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  Params prm;
  st = fill_params(prm, a, pl, ws, reinterpret_cast<uint32_t *>(ws + pl.ws_status));
  if (st != MT_OK) return st;
  // the new rows land in private suffix blocks, which only the suffix decode
  // reads (the prefix kernel reads shared blocks only)
  prm.k_new = k_new;
  prm.v_new = v_new;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cp.use) {
    Cascade &c = cp.c;
    c.rec_ml = reinterpret_cast<float *>(ws + cp.rec_off);
    const size_t slots = (size_t)c.n_ctas + (size_t)c.n_tiles;
    c.rec_o = reinterpret_cast<float *>(ws + cp.rec_off +
                                        ((slots * kPrefixRows * 2 * 4 + 255) & ~(size_t)255));
    prm.casc = c;
    if (c.n_units > 0) {
      PrefixParams pp;
      pp.q = a->q;
      pp.k_pool = static_cast<const uint8_t *>(a->k_pool);
      pp.v_pool = static_cast<const uint8_t *>(a->v_pool);
      pp.table = a->block_table;
      pp.ctx = a->context_lens;
      pp.spans = a->spans;
      pp.kv_map = a->kv_map;
      pp.status = prm.status;
      pp.B = prm.B;
      pp.Hq = prm.Hq;
      pp.Hkv = prm.Hkv;
      pp.G = prm.G;
      pp.bs = prm.bs;
      pp.max_blocks = prm.max_blocks;
      pp.n_phys = prm.n_phys;
      pp.row_bytes = prm.row_bytes;
      pp.qscale = prm.qscale;
      pp.c = c;
      st = launch_prefix(a->fmt, a->head_dim, pl.GP, pp, c.n_ctas, s);
      if (st != MT_OK) return st;
    }
  }
  st = dispatch(prm, pl, a->fmt, s);
  return st == MT_OK ? ok() : st;
}
}  // namespace
}  // namespace mtkv

extern "C" mt_status mt_paged_attn_decode_append(const mt_paged_attn_args *a, const float *k_new,
                                                 const float *v_new, void *workspace,
                                                 size_t workspace_bytes, mt_stream stream) {
  Plan pl;
  mt_status st = make_plan(a, &pl, true);
  if (st != MT_OK) return st;
  if (a->n_seqs == 0) return ok();
  if (!a->q || !a->k_pool || !a->v_pool || !a->block_table || !a->context_lens || !a->out ||
      !k_new || !v_new)
    return fail(MT_ERR_INVALID_ARG, "paged decode with append: null pointer");
  if (!workspace || workspace_bytes < pl.ws_total)
    return fail(MT_ERR_INVALID_ARG,
                "paged decode with append: workspace missing or too small (need " +
                    std::to_string(pl.ws_total) + " bytes)");
  if (!aligned16(a->k_pool) || !aligned16(a->v_pool) || !aligned16(a->q) || !aligned16(a->out) ||
      !aligned16(workspace) || !aligned16(k_new) || !aligned16(v_new))
    return fail(MT_ERR_INVALID_ARG,
                "paged decode with append: q, pools, out, new rows and workspace must be 16-byte "
                "aligned");
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  Params prm;
  st = fill_params(prm, a, pl, ws, reinterpret_cast<uint32_t *>(ws + pl.ws_status));
  if (st != MT_OK) return st;
  prm.k_new = k_new;
  prm.v_new = v_new;
  st = dispatch(prm, pl, a->fmt, reinterpret_cast<cudaStream_t>(stream));
  return st == MT_OK ? ok() : st;
}

// ------------------------------------------------ decode without allocation
//
// Some callers cannot allocate device memory at the moment they decode: code
// running under a pre-sized memory budget that must not grow, plugins and
// other embedders that get no allocator from their host, and callers that
// must not call into the CUDA allocator on this thread (for example while
// another component holds it). They cannot size and pass a workspace, so
// this variant keeps the split-K scratch (sequence offsets and the per-split
// partial results) in a fixed array that lives in the library itself.
//
// Limits and sharing:
//  * The array holds MT_STATIC_SCRATCH_BYTES (8 MiB). Every GPU that loads
//    the library keeps that much device memory for it until the process
//    exits. A call whose scratch would not fit (mt_paged_attn_workspace_bytes
//    larger than the array) is refused with MT_ERR_UNSUPPORTED before
//    anything is launched.
//  * All calls on a device share the one array and leave the last call's
//    partial results in it. No byte of it has to start at zero: every byte
//    a call reads was written earlier in the same call. Two calls whose
//    kernels overlap on the GPU (different streams, no ordering between
//    them) race on the array and may produce wrong results; order them on
//    one stream, or use mt_paged_attn_decode with separate workspaces.
//  * The first call on each device looks the array's device address up
//    (cudaGetSymbolAddress, with that device current) and caches it; make
//    that first call before any stream capture begins. The address is the
//    array's in the device's current context: after cudaDeviceReset (or
//    anything else that destroys and re-creates that context) the cached
//    value is stale and this entry point must not be called again in the
//    process.
//  * The device status word is the caller's `status` (may be NULL), not part
//    of the array.
namespace mtkv {
namespace {

constexpr size_t kStaticScratchBytes = MT_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_decode_scratch on the current device (host code only
// sees a host-side stand-in when it names the array).
mt_status static_scratch(uint8_t **out) {
  static std::mutex mu;
  static void *addr[kMaxDevices] = {};
  int dev = 0;
  mt_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != MT_OK) return st;
  if (dev < 0 || dev >= kMaxDevices)
    return fail(MT_ERR_UNSUPPORTED, "static-scratch decode: device index above 63");
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    st = cuda_check(cudaGetSymbolAddress(&p, g_decode_scratch),
                    "cudaGetSymbolAddress(static decode scratch)");
    if (st != MT_OK) return st;
    addr[dev] = p;
  }
  *out = static_cast<uint8_t *>(addr[dev]);
  return MT_OK;
}

}  // namespace
}  // namespace mtkv

extern "C" mt_status mt_paged_attn_decode_static(const mt_paged_attn_args *a, uint32_t *status,
                                                 mt_stream stream) {
  Plan pl;
  mt_status st = make_plan(a, &pl, true);
  if (st != MT_OK) return st;
  if (pl.ws_total > kStaticScratchBytes)
    return fail(MT_ERR_UNSUPPORTED,
                "static-scratch decode: this call needs " + std::to_string(pl.ws_total) +
                    " bytes of scratch but the library's array holds " +
                    std::to_string(kStaticScratchBytes) +
                    "; use mt_paged_attn_decode with a workspace");
  if (a->n_seqs == 0) return ok();
  if (!a->q || !a->k_pool || !a->v_pool || !a->block_table || !a->context_lens || !a->out)
    return fail(MT_ERR_INVALID_ARG, "static-scratch decode: null pointer");
  if (!aligned16(a->k_pool) || !aligned16(a->v_pool) || !aligned16(a->q) || !aligned16(a->out))
    return fail(MT_ERR_INVALID_ARG, "static-scratch decode: q, pools and out must be 16-byte aligned");
  uint8_t *ws = nullptr;
  st = static_scratch(&ws);
  if (st != MT_OK) return st;
  Params prm;
  st = fill_params(prm, a, pl, ws, status);
  if (st != MT_OK) return st;
  st = dispatch(prm, pl, a->fmt, reinterpret_cast<cudaStream_t>(stream));
  return st == MT_OK ? ok() : st;
}
