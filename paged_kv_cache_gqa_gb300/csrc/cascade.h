// Shared-prefix (cascade) decode: the description shared by the prefix
// kernel, the suffix decode and the combine step.
//
// "Tiered KV cache — architecture", section "The paged-attention block
// model", point 2 (copy-on-write by per-block refcounts: forks of one prompt
// point their block tables at the same physical prefix blocks) and "KV Cache Design — cells,
// format, sessions", section 1 (a sequence reads another's prefix in place
// through its window). When the sequences of a group share their first
// `nblk` block-table entries, the prefix kernel streams each shared block
// once for all of them (their decode queries form the rows of one
// tensor-core tile per KV head); the ordinary decode then reads only each
// sequence's private suffix, and the combine merges both by log-sum-exp.
//
// Work of the prefix kernel: tiles in the order (group, query tile of `tq`
// sequences, KV head); a tile has one unit per prefix block. The units are cut
// into equal contiguous ranges, one per CTA; CTA c writes its share of tile T
// as one partial record in slot c + T (unique: a CTA's tiles increase and
// neighbouring CTAs share at most one tile).
#pragma once

#include <stdint.h>

namespace mtkv {

constexpr int kMaxPrefixGroups = 64;
constexpr int kPrefixRows = 64;  // (sequence, query head) rows of a prefix tile

struct PrefixGroup {
  int s0, s1;  // sequences [s0, s1)
  int nblk;    // shared leading block-table entries
};

struct Cascade {
  int n_groups;  // 0: no cascade
  int tq;        // sequences per tile = kPrefixRows / padded query group
  int gp;        // padded query group (rows per sequence in a tile)
  int n_tiles;
  long long n_units;
  int per;       // units per prefix CTA
  int n_ctas;    // prefix kernel CTAs
  float *rec_ml; // [n_ctas + n_tiles][kPrefixRows][2]  (max, sum), base-2 logits
  float *rec_o;  // [n_ctas + n_tiles][kPrefixRows][D] unnormalised outputs
  PrefixGroup g[kMaxPrefixGroups];
};

__host__ __device__ inline int cascade_qtiles(const Cascade &c, int i) {
  return (c.g[i].s1 - c.g[i].s0 + c.tq - 1) / c.tq;
}

// Unit u -> tile T, group, query tile, KV head, prefix block b.
__host__ __device__ inline void cascade_unit(const Cascade &c, int Hkv, long long u, int &T,
                                             int &grp, int &qt, int &kvh, int &b) {
  int t_base = 0;
  long long u_base = 0;
  for (int i = 0; i < c.n_groups; ++i) {
    const int tiles = cascade_qtiles(c, i) * Hkv;
    const long long units = (long long)tiles * c.g[i].nblk;
    if (u < u_base + units) {
      const long long local = u - u_base;
      const int t_local = (int)(local / c.g[i].nblk);
      b = (int)(local % c.g[i].nblk);
      qt = t_local / Hkv;
      kvh = t_local % Hkv;
      grp = i;
      T = t_base + t_local;
      return;
    }
    t_base += tiles;
    u_base += units;
  }
  T = grp = qt = kvh = b = -1;
}

// Group of sequence s (-1 if none) with its tile, row and unit range for
// query head h: the records of (s, h) are slots c + T, row R, for the CTAs c
// whose unit ranges meet [u0, u0 + nblk).
__host__ __device__ inline int cascade_find(const Cascade &c, int Hkv, int G, int s, int h, int &T,
                                            int &R, long long &u0) {
  int t_base = 0;
  long long u_base = 0;
  for (int i = 0; i < c.n_groups; ++i) {
    const int tiles = cascade_qtiles(c, i) * Hkv;
    if (s >= c.g[i].s0 && s < c.g[i].s1) {
      const int j = s - c.g[i].s0;
      const int t_local = (j / c.tq) * Hkv + h / G;
      T = t_base + t_local;
      R = (j % c.tq) * c.gp + h % G;
      u0 = u_base + (long long)t_local * c.g[i].nblk;
      return i;
    }
    t_base += tiles;
    u_base += (long long)tiles * c.g[i].nblk;
  }
  return -1;
}

// First position of sequence s that the suffix decode reads (0 if none).
__host__ __device__ inline int cascade_skip(const Cascade &c, int s, int bs) {
  for (int i = 0; i < c.n_groups; ++i)
    if (s >= c.g[i].s0 && s < c.g[i].s1) return c.g[i].nblk * bs;
  return 0;
}

}  // namespace mtkv
