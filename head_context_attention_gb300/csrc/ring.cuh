// ring.cuh -- geometry of the emulated 2D mesh: paired-block (zigzag) or
// contiguous placement of ring ranks, the inner/outer double-ring step order,
// and the walk over the key tiles a query tile meets along its ring pass.
//
// [G] "Guide to LoongTrain: 2D Head-Context Parallelism for LLMs":
//   section 2 (Paired-Block Allocation): ring rank r owns blocks r and
//   2*P_seq-1-r of the 2*P_seq blocks;
//   "The Communication Overhead and Causal Imbalance of Ring Attention":
//   query i sees key j only for j <= i.
// [A] abstract: Double-Ring-Attention; the step order used is the nested one
//   (one inner-ring hop per step, one outer-ring hop per inner round).
#pragma once

#include <stdint.h>

namespace loong {

constexpr int kTile = 128;  // rows of a query tile and of a key tile

struct RingGeom {
  int cp, inner, outer;
  int causal;   // 1: query i sees keys j <= i; 0: every key
  int zigzag;   // 1 paired blocks, 0 contiguous
  int blk;      // tokens per block
  int nblocks;  // blocks per sequence: 2*cp or cp
  int ntile;    // key/query tiles per block: ceil(blk / 128)
};

__host__ __device__ inline int ring_src(int c, int t, int inner, int outer) {
  const int o = t / inner, i = t - (t / inner) * inner;
  const int g = c / inner, l = c - (c / inner) * inner;
  return ((g - o + outer) % outer) * inner + (l - i + inner) % inner;
}

// Ring rank that owns natural block b.
__host__ __device__ inline int block_owner(const RingGeom& g, int b) {
  return g.zigzag ? (b < g.cp ? b : 2 * g.cp - 1 - b) : b;
}

// Natural block index of part `part` (0 = A, 1 = B) of ring rank c.
__host__ __device__ inline int rank_block(const RingGeom& g, int c, int part) {
  return part == 0 ? c : 2 * g.cp - 1 - c;
}

__host__ __device__ inline int rank_parts(const RingGeom& g) { return g.zigzag ? 2 : 1; }

// Where a [tokens, heads, d] tensor keeps token t of sequence b, head h, seen
// as the 3-D view [rows, view heads, d] that the TMA maps and the element
// offsets use.
//   natural     [B, S, H, d]: row b*S + t, view head h.
//   rank-major  [B*cp, P, S/cp, H/P, d], the layout of every emulated rank
//               after the Ulysses exchange ([G] "The Scalability Limits of
//               DeepSpeed Ulysses") inside ring rank c: rank c's S/cp tokens
//               (its blocks in part order) for head rank p's H/P heads.  Row
//               ((b*cp + c)*P + p)*(S/cp) + u for the rank-local position u of
//               t, view head h mod H/P.
// A 128-token tile never crosses a block, so its rows are consecutive in
// both layouts.
struct Layout {
  int rank_major;
  int P, cp, zigzag, blk;
  int64_t S;
  int64_t s_rank;  // S / cp, tokens per ring rank

  // rank-local position of natural token t and its ring rank c (t < S < 2^31:
  // a 32-bit division)
  __host__ __device__ int64_t rank_pos(int64_t t, int& c) const {
    const int k = static_cast<int>(t) / blk;
    const int64_t off = t - static_cast<int64_t>(k) * blk;
    if (zigzag && k >= cp) {
      c = 2 * cp - 1 - k;
      return blk + off;
    }
    c = k;
    return off;
  }
  __host__ __device__ int view_heads(int H) const { return rank_major ? H / P : H; }
  // row of (b, t, h) in the view of a tensor with H heads, and its view head
  __host__ __device__ int64_t view_row(int b, int64_t t, int h, int H, int& hc) const {
    if (!rank_major) {
      hc = h;
      return static_cast<int64_t>(b) * S + t;
    }
    const int hpr = H / P;
    const int p = h / hpr;
    hc = h - p * hpr;
    int c;
    const int64_t u = rank_pos(t, c);
    return ((static_cast<int64_t>(b) * cp + c) * P + p) * s_rank + u;
  }
  // rank-major only: the row of (b, t, h) in ring rank `holder`'s plane, at
  // t's rank-local position (where a rank keeps the chunk it has received)
  __host__ __device__ int64_t view_row_held(int b, int64_t t, int h, int H, int holder, int& hc) const {
    const int hpr = H / P;
    const int p = h / hpr;
    hc = h - p * hpr;
    int c;
    const int64_t u = rank_pos(t, c);
    return ((static_cast<int64_t>(b) * cp + holder) * P + p) * s_rank + u;
  }
  // index of the d-vector of (b, t, h), in units of d elements
  __host__ __device__ int64_t vec(int b, int64_t t, int h, int H) const {
    int hc;
    const int64_t r = view_row(b, t, h, H, hc);
    return r * view_heads(H) + hc;
  }
  // rows of the view
  __host__ __device__ int64_t view_rows(int64_t batch) const { return batch * S * (rank_major ? P : 1); }
};

// Key tiles that the query tile (natural block bq, tile qi of that block)
// meets over ring steps [t0, t1), in ring order: step by step, block A then
// block B of the step's source rank, tiles in increasing position.  Causal:
// blocks that lie wholly after bq are skipped and the block bq itself is
// visited up to the diagonal tile qi.  Non-causal: every tile of every block.
struct KvWalk {
  RingGeom g;
  int c, bq, qi, t, t1, part, kt, kt_n, bk;
  int t_first;  // the first step of the walk

  __host__ __device__ void init(const RingGeom& geom, int bq_, int qi_, int t0, int t1_) {
    g = geom;
    bq = bq_;
    qi = qi_;
    c = block_owner(g, bq);
    t_first = t0;
    t = t0;
    t1 = t1_;
    part = 0;
    kt = 0;
    settle();
  }
  __host__ __device__ void settle() {
    while (t < t1) {
      const int j = ring_src(c, t, g.inner, g.outer);
      bk = rank_block(g, j, part);
      kt_n = (!g.causal || bk < bq) ? g.ntile : (bk == bq ? qi + 1 : 0);
      if (kt < kt_n) return;
      kt = 0;
      if (++part == rank_parts(g)) {
        part = 0;
        ++t;
      }
    }
  }
  __host__ __device__ bool done() const { return t >= t1; }
  __host__ __device__ int k0() const { return bk * g.blk + kt * kTile; }
  __host__ __device__ int klen() const {
    const int e = (bk + 1) * g.blk - k0();
    return e < kTile ? e : kTile;
  }
  __host__ __device__ bool diag() const { return g.causal && bk == bq && kt == qi; }
  // The next tile: within the block without recomputing the ring position
  // (the ring arithmetic divides by the ring sizes), else the next block.
  __host__ __device__ void advance() {
    if (++kt < kt_n) return;
    kt = 0;
    if (++part == rank_parts(g)) {
      part = 0;
      ++t;
    }
    settle();
  }
  // Number of tiles of the whole walk, right after init.  Over every ring
  // step each block is visited once, so the count has a closed form: every
  // tile of every earlier block and the diagonal block up to qi (causal), or
  // every tile (non-causal).  A partial range of steps walks a copy.
  __host__ __device__ int total() const {
    if (t_first == 0 && t1 == g.inner * g.outer)
      return g.causal ? bq * g.ntile + qi + 1 : g.nblocks * g.ntile;
    return count();
  }
  // Number of tiles left, walking a copy.
  __host__ __device__ int count() const {
    int n = 0;
    int tt = t;
    int pp = part;
    int first = kt;
    while (tt < t1) {
      const int j = ring_src(c, tt, g.inner, g.outer);
      const int b = rank_block(g, j, pp);
      const int m = (!g.causal || b < bq) ? g.ntile : (b == bq ? qi + 1 : 0);
      if (m > first) n += m - first;
      first = 0;
      if (++pp == rank_parts(g)) {
        pp = 0;
        ++tt;
      }
    }
    return n;
  }
};

// Ring rank that holds source j's K/V at step t (inverse of ring_src in c).
__host__ __device__ inline int ring_dst(int j, int t, int inner, int outer) {
  const int o = t / inner, i = t - (t / inner) * inner;
  const int g = j / inner, l = j - (j / inner) * inner;
  return ((g + o) % outer) * inner + (l + i) % inner;
}

// The (query tile, head) pairs that meet key tile (block bk, tile kt) over
// ring steps [t0, t1), in the order the K/V chunk visits ranks: step by step,
// the destination rank's block A then B, then its query tiles and the G heads
// of the kv group.  Within a block the tiles (and the heads) start at an offset
// `rot`, so that CTAs of neighbouring key tiles, which walk the same blocks at
// the same time, add into different dQ rows.
struct QWalk {
  RingGeom g;
  int G, bk, kt, j, t, t1, part, rot;
  int t_first;  // the first step of the walk
  int qlo, len, k, hk;  // tiles [qlo, ntile) of the current block; position k; head position hk
  int rot_len, rot_g;   // rot reduced modulo len (per block) and modulo G
  int qi, head, bq;

  __host__ __device__ void init(const RingGeom& geom, int G_, int bk_, int kt_, int t0, int t1_, int rot_ = 0) {
    g = geom;
    G = G_;
    bk = bk_;
    kt = kt_;
    j = block_owner(g, bk);
    t_first = t0;
    t = t0;
    t1 = t1_;
    part = 0;
    rot = rot_ < 0 ? 0 : rot_;
    rot_g = rot % G;
    next_block(true);
  }
  // Settle on the first (tile, head) of the current or next block that sees bk.
  __host__ __device__ void next_block(bool same) {
    if (!same) step_part();
    while (t < t1) {
      const int c = ring_dst(j, t, g.inner, g.outer);
      bq = rank_block(g, c, part);
      qlo = (!g.causal || bk < bq) ? 0 : (bk == bq ? kt : g.ntile);
      len = g.ntile - qlo;
      if (len > 0) {
        k = 0;
        hk = 0;
        rot_len = rot % len;
        set();
        return;
      }
      step_part();
    }
  }
  __host__ __device__ void step_part() {
    if (++part == rank_parts(g)) {
      part = 0;
      ++t;
    }
  }
  // qi = qlo + (k + rot) mod len, head = (hk + rot) mod G, without dividing
  // (k < len, hk < G)
  __host__ __device__ void set() {
    const int x = k + rot_len;
    qi = qlo + (x >= len ? x - len : x);
    const int y = hk + rot_g;
    head = y >= G ? y - G : y;
  }
  __host__ __device__ bool done() const { return t >= t1; }
  __host__ __device__ void advance() {
    if (++hk < G) {
      set();
      return;
    }
    hk = 0;
    if (++k < len) {
      set();
      return;
    }
    next_block(false);
  }
  __host__ __device__ int q0() const { return bq * g.blk + qi * kTile; }
  __host__ __device__ int qlen() const {
    const int e = (bq + 1) * g.blk - q0();
    return e < kTile ? e : kTile;
  }
  __host__ __device__ bool diag() const { return g.causal && bq == bk && qi == kt; }
  // Number of (tile, head) pairs of the whole walk, right after init: over
  // every ring step each query block is visited once (closed form: every
  // tile of every later block and the key tile's own block from kt on, or
  // every tile when non-causal), else a copy is walked.
  __host__ __device__ int total() const {
    if (t_first == 0 && t1 == g.inner * g.outer)
      return G * (g.causal ? (g.nblocks - 1 - bk) * g.ntile + g.ntile - kt : g.nblocks * g.ntile);
    return count();
  }
  __host__ __device__ int count() const {
    int n = 0;
    for (int tt = t; tt < t1; ++tt) {
      const int c = ring_dst(j, tt, g.inner, g.outer);
      for (int pp = 0; pp < rank_parts(g); ++pp) {
        const int b = rank_block(g, c, pp);
        if (!g.causal || bk < b) n += g.ntile;
        else if (bk == b) n += g.ntile - kt;
      }
    }
    return n * G;
  }
};

}  // namespace loong
