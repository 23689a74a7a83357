// Multi-query (prefill) paged attention on the 5th-generation tensor cores
// (tcgen05, tensor-memory accumulators), for f16 pools.
//
// What is computed — exactly what prefill.cu computes (see there): for query
// row i of sequence s at position ctx - n + j, softmax-weighted V over the
// positions t <= its own, t < ctx, not in a hole, inside its window ("Tiered
// KV cache — architecture", sections "The paged-attention block model" and
// "Kernel dispatch"; "KV Cache Design — cells, format, sessions", section 1).
//
// How (GB300): a tile is 128 (query, head) rows of one KV head — one row per
// thread of a 4-warp CTA, which is also that row's tensor-memory lane — and
// the sequence's positions up to the tile's last query, in chunks of 64
// tokens. Per chunk:
//   1. the chunk's K and V head slices are copied (cp.async, 16 B) into
//      128-byte-swizzled shared tiles, [token][64 dims] per half head; holes
//      and rows past the context are zero-filled (no read);
//   2. one thread issues S = Q_hi K^T + Q_lo K^T (M = 128, N = 64, f16 in,
//      f32 accumulated in tensor memory; q = Q_hi + Q_lo to ~2^-22, so scores
//      keep float32 accuracy) and commits to an mbarrier;
//   3. every thread loads its row of S, masks it, and runs its own online
//      softmax in registers (no cross-thread reduction); the output row in
//      tensor memory is rescaled only when the running maximum grows by more
//      than 2^8 (probabilities then stay below 256, exact in f16);
//   4. the probabilities go to a swizzled P tile (f16) and one thread issues
//      O += P V (N = head_dim; V read MN-major straight from its tile).
// Chunks are staged three ahead; a tile's output is normalised once at the
// end. CTAs take whole tiles round-robin (no split-K combine).
#include <limits.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "mma.cuh"
#include "prefill.h"
#include "tc.cuh"

namespace mtkv {
namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kTcRows = 128;    // rows per tile = threads per CTA
constexpr int kChunk = 64;      // tokens per chunk
constexpr int kTcStages = 4;
constexpr int kOCol = 2 * 64;        // S double buffer: columns [0, 64), [64, 128); O: [128, 128 + d)
constexpr uint32_t kTmemCols = 256;

template <int D>
struct TcCfg {
  static constexpr int HALVES = D / 64;                 // 64-dim halves of a head
  static constexpr int QB = HALVES * kTcRows * 128;     // one Q tile (hi or lo)
  static constexpr int PB = kTcRows * 128;              // P tile: 128 rows x 64 tokens
  static constexpr int KVB = HALVES * kChunk * 128;     // K (or V) of one chunk
  static constexpr int STAGE = 2 * KVB;
  static constexpr int SMEM = 1024 + 2 * QB + PB + kTcStages * STAGE;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t n) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 2^x by the hardware approximation (relative error ~2^-22, 2^-inf = 0):
// far below the f16 rounding the probabilities get right after.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
  tl.nch = reach > 0 ? (reach + kChunk - 1) / kChunk : 0;
  return true;
}

// Block ids of chunk `ch` (block k of the chunk -> ids[k]; -1: a hole, a
// flagged id or past the context), loaded by the first 64 / bs threads.
__device__ __forceinline__ void load_chunk_ids(const PrefillParams &p, const Tile &tl, int ch,
                                               int *ids) {
  const int nb = kChunk / p.bs;
  if ((int)threadIdx.x < nb) {
    const int pos = ch * kChunk + (int)threadIdx.x * p.bs;
    int phys = -1;
    if (ch < tl.nch && pos < tl.c) {
      phys = p.table[(size_t)tl.s * p.max_blocks + pos / p.bs];
      if (phys < -1 || (phys >= 0 && (long long)phys >= p.n_phys)) {
        report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
        phys = -1;
      }
    }
    ids[threadIdx.x] = phys;
  }
}

// Copy chunk `ch` of the tile's KV head into ring slot `slot` (every thread
// issues its share; one commit group per call, empty past the last chunk).
// Rows of holes and past the context are zero-filled without a read. Thread
// t always moves 16-byte column t % CPR of rows t / CPR + (128 / CPR) k, so
// its shared-memory column and swizzle are fixed.
template <int D>
__device__ __forceinline__ void issue_chunk(const PrefillParams &p, const Tile &tl, int ch,
                                            const int *ids, uint8_t *ring, int slot,
                                            int bs_shift) {
  using C = TcCfg<D>;
  constexpr int CPR = D * 2 / 16;        // 16-byte columns per head row
  constexpr int RSTEP = kTcRows / CPR;   // rows between a thread's items
  constexpr int ITEMS = kChunk / RSTEP;
  if (ch < tl.nch) {
    const int cc = threadIdx.x % CPR, t0 = threadIdx.x / CPR;
    const uint32_t base = smem_u32(ring + (size_t)slot * C::STAGE) +
                          (uint32_t)((cc >> 3) * kChunk * 128) + (uint32_t)t0 * 128 +
                          (uint32_t)(((cc & 7) ^ (t0 & 7)) << 4);
    const size_t col = (size_t)tl.kvh * D * 2 + (size_t)cc * 16;
    const int pos0 = ch * kChunk, bmask = (1 << bs_shift) - 1;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      const int t = t0 + RSTEP * k;  // RSTEP is a multiple of 8: the swizzle is unchanged
      const int pos = pos0 + t;
      const int phys = ids[t >> bs_shift];
      const bool ok = phys >= 0 && pos < tl.c;
      const size_t g =
          ok ? (((size_t)phys << bs_shift) + (pos & bmask)) * (size_t)p.row_bytes + col : 0;
      const uint32_t dst = base + (uint32_t)(RSTEP * k * 128);
      cp_async16(dst, p.k_pool + g, ok ? 16u : 0u);
      cp_async16(dst + C::KVB, p.v_pool + g, ok ? 16u : 0u);
    }
  }
  cp_commit();
}

template <int D, int GP>
__global__ void __launch_bounds__(kTcRows, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using C = TcCfg<D>;
  constexpr int TQ = kTcRows / GP;
  constexpr int R_RUNS = MT_KV_MAP_MAX_SPANS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int ts[kMaxPrefillSeqs + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar_s[2], bar_pv;
  __shared__ int ids_s[kTcStages][4];  // block ids of the staged chunks, by slot
  __shared__ int abort_s;
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *qhi = base;
  uint8_t *qlo = base + C::QB;
  uint8_t *pt = base + 2 * C::QB;
  uint8_t *ring = pt + C::PB;
  pdl_enter();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // tile offsets: ceil(n_s / TQ) query tiles per sequence, times Hkv
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
    mbar_init(&bar_s[0], 1);
    mbar_init(&bar_s[1], 1);
    mbar_init(&bar_pv, 1);
    abort_s = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int n_tiles = ts[p.B];
  if ((int)blockIdx.x >= n_tiles) return;
  if (warp == 0) tc::alloc(&tmem_slot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's lanes
  constexpr uint32_t idesc_s = tc::idesc_f16(kTcRows, kChunk, false);
  constexpr uint32_t idesc_o = tc::idesc_f16(kTcRows, D, true);
  uint32_t ph_pv = 0;
  const int bs_shift = p.bs == 32 ? 5 : 4;
  uint32_t n_s0 = 0, n_s1 = 0;  // completions consumed per S buffer (their wait parity)
  bool ok_run = true;
  const uint64_t wait_ns = 2000000000ull;

  for (int t = blockIdx.x; ok_run; t += gridDim.x) {
    Tile tl;
    if (!tile_of<GP>(p, ts, n_tiles, t, tl)) break;
    // ---- this thread's row: (query j, head hg)
    const int j = tl.qt * TQ + tid / GP, hg = tid % GP;
    const int i = p.q_start[tl.s] + j;
    const int pos_q = tl.c - tl.n + j;
    const bool row_in = j < tl.n && hg < p.G && i >= 0 && i < p.n_tok;
    if (j < tl.n && hg < p.G && !row_in) report(p.status, MT_STATUS_BIT_DEVICE_CHECK);
    const bool row_ok = row_in && pos_q >= 0;
    int lo = 0, hi = row_ok ? min(pos_q + 1, tl.c) : 0;
    if (row_ok && p.spans) {
      lo = max(p.spans[2 * i], 0);
      hi = min(hi, p.spans[2 * i + 1]);
    }
    int ra[R_RUNS], re[R_RUNS];
    if (p.kv_map) {
#pragma unroll
      for (int r = 0; r < R_RUNS; ++r) {
        ra[r] = re[r] = 0;
        if (row_ok) {
          const int32_t *rp = p.kv_map + ((size_t)i * R_RUNS + r) * 2;
          ra[r] = max(rp[0], 0);
          re[r] = min(rp[0] + rp[1], hi);
        }
      }
    }
    // ---- the row's query as a high / low f16 pair in the two Q tiles
    {
      const float *qrow = p.q + ((size_t)(row_ok ? i : 0) * p.Hq + (size_t)tl.kvh * p.G + hg) * D;
#pragma unroll 4
      for (int e = 0; e < D; e += 8) {
        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
        if (row_ok) {
          x0 = *reinterpret_cast<const float4 *>(qrow + e);
          x1 = *reinterpret_cast<const float4 *>(qrow + e + 4);
        }
        uint32_t h[4], l[4];
        const float qs = p.qscale;
        split_h2(x0.x * qs, x0.y * qs, h[0], l[0]);
        split_h2(x0.z * qs, x0.w * qs, h[1], l[1]);
        split_h2(x1.x * qs, x1.y * qs, h[2], l[2]);
        split_h2(x1.z * qs, x1.w * qs, h[3], l[3]);
        const uint32_t off = (uint32_t)((e >> 6) * kTcRows * 128) + tc::sw128(tid, (e & 63) >> 3);
        *reinterpret_cast<uint4 *>(qhi + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(qlo + off) = make_uint4(l[0], l[1], l[2], l[3]);
      }
    }
    float m_run = -INFINITY, l_run = 0.f;

    // ---- chunks: S(ch+1) is computed by the tensor cores while the threads
    // run the softmax of chunk ch (two S buffers, one mbarrier each)
    load_chunk_ids(p, tl, 0, ids_s[0]);
    load_chunk_ids(p, tl, 1, ids_s[1]);
    load_chunk_ids(p, tl, 2, ids_s[2]);
    load_chunk_ids(p, tl, 3, ids_s[3]);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kTcStages - 1; ++k) issue_chunk<D>(p, tl, k, ids_s[k], ring, k, bs_shift);
    auto issue_s = [&](int x) {
      // S(x) = Q_hi K^T + Q_lo K^T into S buffer x % 2 (one thread)
      const uint8_t *kt = ring + (size_t)(x % kTcStages) * C::STAGE;
      const uint32_t dcol = tmem + (uint32_t)((x & 1) * 64);
#pragma unroll
      for (int hf = 0; hf < C::HALVES; ++hf)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t qo = (uint32_t)(hf * kTcRows * 128 + kk * 32);
          const uint64_t bd = tc::desc_sw128(smem_u32(kt) + hf * kChunk * 128 + kk * 32, 16, 1024);
          tc::mma_f16(dcol, tc::desc_sw128(smem_u32(qhi) + qo, 16, 1024), bd, idesc_s,
                      hf + kk > 0);
          tc::mma_f16(dcol, tc::desc_sw128(smem_u32(qlo) + qo, 16, 1024), bd, idesc_s, true);
        }
      tc::commit(&bar_s[x & 1]);
    };
    for (int ch = 0; ch < tl.nch; ++ch) {
      // chunks ch and ch+1 staged (groups: S-1 in the prologue, one per iteration)
      cp_wait<kTcStages - 3>();
      tc::fence_proxy_shared();  // this thread's copies (and Q / P writes) -> async proxy
      tc::fence_before();
      __syncthreads();
      tc::fence_after();
      if (tid == 0) {
        if (ch == 0) issue_s(0);
        if (ch + 1 < tl.nch) issue_s(ch + 1);
      }
      // a wait that runs out is carried to the next CTA barrier, where every
      // thread leaves together (no thread may skip a barrier the others reach)
      bool fine = mbar_wait_bounded(&bar_s[ch & 1], ((ch & 1) ? n_s1 : n_s0) & 1u, &abort_s,
                                    wait_ns);
      if (ch & 1) ++n_s1; else ++n_s0;
      tc::fence_after();
      float sv[kChunk];
#pragma unroll
      for (int c16 = 0; c16 < kChunk; c16 += 16) {
        float v[16];
        tc::ld16(t_row + (uint32_t)((ch & 1) * 64) + c16, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) sv[c16 + e] = v[e];
      }
      tc::wait_ld();
      // ---- mask: positions of this chunk the row may read
      const int pos0 = ch * kChunk;
      uint64_t mk = 0;
      if (p.kv_map) {
#pragma unroll
        for (int r = 0; r < R_RUNS; ++r) {
          const int a = max(ra[r] - pos0, 0), b = min(re[r] - pos0, kChunk);
          if (b > a) mk |= (b >= 64 ? ~0ull : ((1ull << b) - 1ull)) & ~((1ull << a) - 1ull);
        }
      } else {
        const int a = max(lo - pos0, 0), b = min(hi - pos0, kChunk);
        if (b > a) mk = (b >= 64 ? ~0ull : ((1ull << b) - 1ull)) & ~((1ull << a) - 1ull);
      }
      // holes (and flagged ids) read as -infinity
      {
        const int *ids = ids_s[ch % kTcStages];
        const uint64_t bmask = p.bs >= 64 ? ~0ull : ((1ull << p.bs) - 1ull);
        for (int k = 0; k * p.bs < kChunk; ++k)
          if (ids[k] < 0) mk &= ~(bmask << (k * p.bs));
      }
      // most chunks are wholly readable: only partial ones pay for the mask
      if (mk != ~0ull) {
        const uint32_t m0 = (uint32_t)mk, m1 = (uint32_t)(mk >> 32);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          sv[e] = (m0 & (1u << e)) ? sv[e] : -INFINITY;
          sv[e + 32] = (m1 & (1u << e)) ? sv[e + 32] : -INFINITY;
        }
      }
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // 4 independent chains
#pragma unroll
      for (int e = 0; e < kChunk; ++e) mq[e & 3] = fmaxf(mq[e & 3], sv[e]);
      const float mloc = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      // ---- the previous P.V has finished: O, the P tile and the previous slot are free
      if (ch > 0) {
        fine = mbar_wait_bounded(&bar_pv, ph_pv, &abort_s, wait_ns) && fine;
        ph_pv ^= 1u;
        tc::fence_after();
      }
      issue_chunk<D>(p, tl, ch + kTcStages - 1, ids_s[(ch + kTcStages - 1) % kTcStages], ring,
                     (ch + kTcStages - 1) % kTcStages, bs_shift);
      // ---- online softmax, rescaling O only when the maximum grows past 2^8
      const float m_new = fmaxf(m_run, mloc);
      float scale_o = 1.f;
      if (m_new != -INFINITY && (m_run == -INFINITY || m_new > m_run + 8.f)) {
        scale_o = m_run == -INFINITY ? 1.f : exp2f(m_run - m_new);
        l_run *= scale_o;
        m_run = m_new;
      }
      if (ch > 0 && __any_sync(kAll, scale_o != 1.f)) {
#pragma unroll 1
        for (int c16 = 0; c16 < D; c16 += 16) {
          float v[16];
          tc::ld16(t_row + kOCol + c16, v);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= scale_o;
          tc::st16(t_row + kOCol + c16, v);
        }
        tc::wait_st();
      }
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      const float mr = m_run == -INFINITY ? 0.f : m_run;  // all sv are -inf then: p = 0
#pragma unroll
      for (int e = 0; e < kChunk; e += 8) {
        uint32_t h[4];
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const float a = ex2(sv[e + 2 * k2] - mr);
          const float b = ex2(sv[e + 2 * k2 + 1] - mr);
          ls[k2] += a + b;
          h[k2] = h2_bits(__floats2half2_rn(a, b));
        }
        *reinterpret_cast<uint4 *>(pt + tc::sw128(tid, e >> 3)) = make_uint4(h[0], h[1], h[2], h[3]);
      }
      l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tc::fence_proxy_shared();
      tc::fence_before();
      if (!__syncthreads_and(fine)) {
        ok_run = false;
        break;
      }
      // every thread has read this chunk's block ids: the slot takes those of
      // chunk ch + S (copied in the next iteration)
      load_chunk_ids(p, tl, ch + kTcStages, ids_s[ch % kTcStages]);
      if (tid == 0) {
        tc::fence_after();
        // O += P V (V MN-major: LBO = the distance between its 64-dim halves)
        const uint8_t *vt = ring + (size_t)(ch % kTcStages) * C::STAGE + C::KVB;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_f16(tmem + kOCol, tc::desc_sw128(smem_u32(pt) + kk * 32, 16, 1024),
                      tc::desc_sw128(smem_u32(vt) + kk * 2048, kChunk * 128, 1024), idesc_o,
                      ch > 0 || kk > 0);
        tc::commit(&bar_pv);
      }
    }
    cp_wait<0>();
    if (!ok_run) break;
    // ---- the last P.V, then the normalised row
    bool fine = true;
    if (tl.nch > 0) {
      fine = mbar_wait_bounded(&bar_pv, ph_pv, &abort_s, wait_ns);
      ph_pv ^= 1u;
      tc::fence_after();
    }
    if (!__syncthreads_and(fine)) {
      ok_run = false;
      break;
    }
    const bool any = l_run > 0.f;
    const float inv = any ? 1.f / l_run : 0.f;
    float *dst = row_in ? p.out + ((size_t)i * p.Hq + (size_t)tl.kvh * p.G + hg) * D : nullptr;
#pragma unroll 1
    for (int c16 = 0; c16 < D; c16 += 16) {
      float v[16];
      if (tl.nch > 0) {
        tc::ld16(t_row + kOCol + c16, v);
        tc::wait_ld();
      }
      if (dst) {
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4 *>(dst + c16 + e) =
              tl.nch > 0 && any
                  ? make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (row_in && p.lse)
      p.lse[(size_t)i * p.Hq + (size_t)tl.kvh * p.G + hg] =
          any ? (m_run + log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
    // every thread is done with tensor memory and the shared tiles of this
    // tile before the next one overwrites them
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  }
  if (!ok_run && tid == 0) report(p.status, MT_STATUS_BIT_TIMEOUT);
  cp_wait<0>();
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, kTmemCols);
}

template <int D, int GP>
mt_status launch_t(const PrefillParams &p, int n_ctas, cudaStream_t s) {
  static int configured_dev = -1;
  auto kern = prefill_tc_kernel<D, GP>;
  constexpr int smem = TcCfg<D>::SMEM;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    mt_status st =
        cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                   "cudaFuncSetAttribute(prefill tc smem)");
    if (st != MT_OK) return st;
    configured_dev = dev;
  }
  return cuda_check(launch_pdl(kern, dim3(n_ctas), dim3(kTcRows), smem, s, p),
                    "prefill tc kernel launch");
}

template <int D>
mt_status launch_d(int gp, const PrefillParams &p, int n_ctas, cudaStream_t s) {
  switch (gp) {
    case 1: return launch_t<D, 1>(p, n_ctas, s);
    case 2: return launch_t<D, 2>(p, n_ctas, s);
    case 4: return launch_t<D, 4>(p, n_ctas, s);
    default: return launch_t<D, 8>(p, n_ctas, s);
  }
}

}  // namespace

bool prefill_tc_supported(mt_kv_format fmt, int head_dim, int block_size) {
  return fmt == MT_KV_F16 && (head_dim == 64 || head_dim == 128) &&
         (block_size == 16 || block_size == 32);
}

mt_status launch_prefill_tc(const PrefillParams &p, int head_dim, int gp, int n_ctas,
                            cudaStream_t stream) {
  return head_dim == 64 ? launch_d<64>(gp, p, n_ctas, stream)
                        : launch_d<128>(gp, p, n_ctas, stream);
}

}  // namespace mtkv
