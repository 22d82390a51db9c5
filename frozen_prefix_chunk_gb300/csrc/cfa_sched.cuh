// Work decomposition shared by the host planner and the kernels.
//
// Query rows are packed GQA-style: a query tile holds `tpt` consecutive chunk
// tokens times the g = Hq/Hkv query heads that read one KV head, row
// r = token_local * g + head_local (rows = tpt * g <= 128).  Every row of a
// tile therefore reads the same K/V tiles, and the causal edge of a tile spans
// only tpt tokens.
//
// A query block is q_per_cta consecutive query tiles of one (window, KV head).
// Its keys are walked as one list of 128-row tiles: the ceil(Lp / 128) prefix
// tiles first, then the chunk tiles some row of the block can see (chunk key
// j is visible to token t iff j <= t; the whole prefix is visible).
//
// Stream-K schedule.  The iterations (query block, key tile) are numbered
// window-major, then KV head, then query block, then key tile; W is their
// total.  A persistent grid of G CTAs gives CTA c the contiguous range
// [floor(c W / G), floor((c+1) W / G)), so every CTA does the same amount of
// tensor work whatever the window lengths.  A CTA walks its range as
// segments, one per query block it touches.  A segment that covers its whole
// block writes the final outputs; a block cut by CTA boundaries leaves one
// partial per CTA, in slot 1 of the CTA holding its start and slot 0 of the
// others, and a merge kernel combines them in CTA order (deterministic).
// With Tiling::nrow > 1 (row mode, below) the same scheme runs once per
// schedule row, over that row's own CTAs.
// Every CTA scans the per-window work itself in its prologue (plan_schedule
// below); the first CTA of each schedule row also stores the row's prefix
// array win_prefix[row][b] (int64, [nrow][batch + 1]) for the merge kernels
// that run afterwards.
#pragma once

#include <stdint.h>

#ifndef __CUDACC__
// host-only build of the schedule logic (the CPU schedule test)
#define __host__
#define __device__
#endif

namespace cfa {

constexpr int kTileM = 128;  // query rows per tile (TMEM lanes)
constexpr int kTileN = 128;  // keys per tile

struct Tiling {
  int g;          // query heads per KV head
  int tpt;        // chunk tokens per query tile
  int rows;       // valid rows per query tile = tpt * g
  int q_per_cta;  // query tiles per query block
  int grid;       // persistent CTAs (G)
  int setup;      // virtual iterations charged at the start of every query block
  int nrow;       // schedule rows: 1, or (row mode) the query blocks of every window
};

// Row mode.  With nrow > 1 every window has nrow query blocks, and the
// schedule is nrow independent stream-K schedules over grid / nrow CTAs each:
// row r holds block r of every (window, KV head), CTAs r * grid / nrow on.
// The rows have the same layout (the same windows and heads in the same
// order, the same prefix key tiles), so CTA j of every row reads the same key
// tiles of the same head at about the same time: the blocks that share K/V
// run in lockstep and a tile is read from DRAM about once, even when the
// heads' K/V is far larger than L2.  With nrow = 1 the iterations are one
// schedule, window-major, then KV head, then query block.
__host__ __device__ inline int row_grid(const Tiling& tl) { return tl.grid / tl.nrow; }

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// The host-side sizes of a call: they size the grids, the TMA maps, the
// output strides and the workspace, so the device cu_seqlens must agree with
// them before any kernel derives a row index from a window.
struct SeqLimits {
  int total_lp, total_lc;  // cu_seqlens_prefix[batch], cu_seqlens_chunk[batch]
  int max_lp, max_lc;      // longest window
};

// Window b of the device cu_seqlens agrees with the host sizes: both arrays
// start at 0 and end at total_lp / total_lc, and the window's prefix and
// chunk lengths lie in [0, max_lp] and [0, max_lc].  When every window
// passes, both arrays are non-decreasing from 0 to their totals, so every row
// a window spans lies inside the tensors the host described, and every
// window is covered by the grids sized from the maxima.
__host__ __device__ inline bool window_valid(const int32_t* cu_p, const int32_t* cu_c, int b,
                                             int batch, const SeqLimits& s) {
  const long long p0 = cu_p[b], p1 = cu_p[b + 1], c0 = cu_c[b], c1 = cu_c[b + 1];
  if (p1 < p0 || p1 - p0 > s.max_lp || c1 < c0 || c1 - c0 > s.max_lc) return false;
  if (b == 0 && (p0 != 0 || c0 != 0)) return false;
  if (b == batch - 1 && (p1 != s.total_lp || c1 != s.total_lc)) return false;
  return true;
}

// All windows (the host-side test and a reference for the device scans).
__host__ __device__ inline bool seqlens_valid(const int32_t* cu_p, const int32_t* cu_c, int batch,
                                              const SeqLimits& s) {
  if (batch < 1) return false;
  for (int b = 0; b < batch; ++b)
    if (!window_valid(cu_p, cu_c, b, batch, s)) return false;
  return true;
}

// Key tiles seen by a query block whose first token is t0 and which spans
// `tok_blk` tokens, in a window with lp prefix rows and lc chunk rows.
__host__ __device__ inline int block_key_tiles(int lp, int lc, int t0, int tok_blk) {
  const int t_hi = (t0 + tok_blk < lc) ? (t0 + tok_blk) : lc;
  return ceil_div(lp, kTileN) + ceil_div(t_hi, kTileN);
}

__host__ __device__ inline int blocks_of_window(const Tiling& tl, int lc) {
  return lc > 0 ? ceil_div(lc, tl.q_per_cta * tl.tpt) : 0;
}

// Iterations charged to query block qb: its key tiles plus tl.setup virtual
// ones at its start.  They stand for the fixed cost of taking up a block in a
// CTA (its Q load, the epilogue of the block before, the pipeline refill), so
// that a CTA whose range crosses a block start gets fewer key tiles and all
// CTAs finish together.  Virtual iterations do no work.
__host__ __device__ inline int block_iters(const Tiling& tl, int lp, int lc, int qb) {
  const int tok_blk = tl.q_per_cta * tl.tpt;
  return tl.setup + block_key_tiles(lp, lc, qb * tok_blk, tok_blk);
}

// Iterations of one KV head's query blocks in a window.
__host__ __device__ inline long long head_work(const Tiling& tl, int lp, int lc) {
  long long w = 0;
  for (int qb = 0, nb = blocks_of_window(tl, lc); qb < nb; ++qb) w += block_iters(tl, lp, lc, qb);
  return w;
}

// Iterations of one KV head's share of a window in schedule row `row`: all
// its query blocks (nrow = 1), or block `row` alone (row mode).
__host__ __device__ inline long long head_work_row(const Tiling& tl, int lp, int lc, int row) {
  if (tl.nrow <= 1) return head_work(tl, lp, lc);
  return row < blocks_of_window(tl, lc) ? block_iters(tl, lp, lc, row) : 0;
}

// The schedule row holding query block qb.
__host__ __device__ inline int row_of_block(const Tiling& tl, int qb) {
  return tl.nrow > 1 ? qb : 0;
}

// Iterations [*first, *end) holding the key tiles of query block (b, hk, qb),
// given the window's first iteration w0 in the block's schedule row (its
// virtual iterations come before *first).
__host__ __device__ inline void block_span(const Tiling& tl, long long w0, int hk, int qb, int lp,
                                           int lc, long long* first, long long* end) {
  long long bs = w0 + (long long)hk * head_work_row(tl, lp, lc, row_of_block(tl, qb));
  if (tl.nrow <= 1)
    for (int q = 0; q < qb; ++q) bs += block_iters(tl, lp, lc, q);
  *first = bs + tl.setup;
  *end = bs + block_iters(tl, lp, lc, qb);
}

// First iteration of CTA c, and the CTA that holds iteration x.
__host__ __device__ inline long long cta_begin(long long c, long long W, int G) {
  return c * W / G;
}
__host__ __device__ inline int cta_of(long long x, long long W, int G) {
  return (int)(((x + 1) * G - 1) / W);
}

// One contiguous piece of a CTA's range inside one query block.
struct Segment {
  int b, hk, qb;         // the query block
  int p0, lp, c0, lc;    // its window
  int n_kt;              // key tiles of the block
  int t_begin, t_end;    // key tiles [t_begin, t_end) of this segment
  int nq;                // query tiles of the block that hold rows
  bool head;             // the block started in an earlier CTA
  bool tail;             // the block continues in a later CTA
};

// Walks a CTA's iteration range segment by segment.  Every role of the CTA
// runs its own copy and sees the same sequence.  ROW selects row mode at
// compile time (Tiling::nrow > 1), so that the one-row kernels carry no row
// logic (their walker state lives in registers through the inner loops).
template <bool ROW>
struct SegmentWalkerT {
  const int32_t* cu_p;
  const int32_t* cu_c;
  int batch, hkv;
  Tiling tl;
  long long cur, end;
  int b, hk, qb, tile;  // in row mode qb stays the CTA's schedule row

  // Start at CTA `cta`'s first iteration: window b0 (whose first iteration
  // is pre_b0) of its row's schedule, which has `total` iterations.
  __host__ __device__ void init(const int32_t* cp, const int32_t* cc, int nb, int nkv,
                                const Tiling& t, int cta, long long total, int b0,
                                long long pre_b0) {
    cu_p = cp;
    cu_c = cc;
    batch = nb;
    hkv = nkv;
    tl = t;
    if constexpr (ROW) {
      const int rg = row_grid(t), row = cta / rg;
      cur = cta_begin(cta % rg, total, rg);
      end = cta_begin(cta % rg + 1, total, rg);
      if (cur >= end) return;
      b = b0;
      const int lp = cu_p[b + 1] - cu_p[b], lc = cu_c[b + 1] - cu_c[b];
      const long long hw = head_work_row(tl, lp, lc, row);
      long long o = cur - pre_b0;
      hk = (int)(o / hw);
      o -= (long long)hk * hw;
      qb = row;
      tile = (int)o;
    } else {
      cur = cta_begin(cta, total, t.grid);
      end = cta_begin(cta + 1, total, t.grid);
      if (cur >= end) return;
      b = b0;
      const int lp = cu_p[b + 1] - cu_p[b], lc = cu_c[b + 1] - cu_c[b];
      const long long hw = head_work(tl, lp, lc);
      long long o = cur - pre_b0;
      hk = (int)(o / hw);
      o -= (long long)hk * hw;
      qb = 0;
      for (;;) {
        const int nk = block_iters(tl, lp, lc, qb);
        if (o < nk) break;
        o -= nk;
        ++qb;
      }
      tile = (int)o;  // iteration within the block, virtual ones first
    }
  }

  // The next segment with key tiles; blocks of which this CTA holds only
  // virtual iterations are passed over.
  __host__ __device__ bool next(Segment& s) {
    while (cur < end) {
      const int tok_blk = tl.q_per_cta * tl.tpt;
      s.b = b;
      s.hk = hk;
      s.qb = qb;
      s.p0 = cu_p[b];
      s.lp = cu_p[b + 1] - s.p0;
      s.c0 = cu_c[b];
      s.lc = cu_c[b + 1] - s.c0;
      const int ni = block_iters(tl, s.lp, s.lc, qb);
      s.n_kt = ni - tl.setup;
      const long long left = end - cur;
      const int v_end = (left < (long long)(ni - tile)) ? tile + (int)left : ni;
      s.t_begin = tile > tl.setup ? tile - tl.setup : 0;
      s.t_end = v_end - tl.setup;
      s.nq = ceil_div(s.lc - qb * tok_blk, tl.tpt);
      if (s.nq > tl.q_per_cta) s.nq = tl.q_per_cta;
      s.head = s.t_begin > 0;
      s.tail = s.t_end < s.n_kt;
      cur += v_end - tile;
      tile = 0;
      if constexpr (ROW) {
        // the same block of the next head or window
        if (++hk >= hkv) {
          hk = 0;
          do {
            ++b;
          } while (b < batch &&
                   head_work_row(tl, cu_p[b + 1] - cu_p[b], cu_c[b + 1] - cu_c[b], qb) == 0);
        }
      } else {
        // the next query block
        if (++qb >= blocks_of_window(tl, s.lc)) {
          qb = 0;
          if (++hk >= hkv) {
            hk = 0;
            do {
              ++b;
            } while (b < batch && cu_c[b + 1] - cu_c[b] == 0);
          }
        }
      }
      if (s.t_end > s.t_begin) return true;
    }
    return false;
  }
};

using SegmentWalker = SegmentWalkerT<false>;
using RowSegmentWalker = SegmentWalkerT<true>;

// The CTAs holding parts of the block whose iterations are [bs, be), in CTA
// order: the one holding bs, then every later one up to the one holding
// be - 1 whose range is not empty (ranges are only empty when there are fewer
// iterations than CTAs).  Returns the count; 0 when one CTA holds the whole
// block.  `parts` has room for `cap` entries.
__host__ __device__ inline int block_parts(long long bs, long long be, long long total, int G,
                                           int* parts, int cap) {
  const int cf = cta_of(bs, total, G), cl = cta_of(be - 1, total, G);
  if (cf == cl) return 0;
  int n = 0;
  for (int c = cf; c <= cl && n < cap; ++c) {
    if (c > cf && total < G && cta_begin(c, total, G) == cta_begin(c + 1, total, G)) continue;
    parts[n++] = c;
  }
  return n;
}

// The same part list in closed form, for a block with iterations [bs, be):
// the number of parts (0 when one CTA holds the whole block) and the CTA
// holding part j.  With total >= G every CTA holds an iteration, so the parts
// are the consecutive CTAs from the one holding bs; with total < G every CTA
// holds at most one, so part j is the CTA holding iteration bs + j.
__host__ __device__ inline int part_count(long long bs, long long be, long long total, int G) {
  const int cf = cta_of(bs, total, G), cl = cta_of(be - 1, total, G);
  if (cf == cl) return 0;
  return total >= G ? cl - cf + 1 : (int)(be - bs);
}
__host__ __device__ inline int part_cta(long long bs, long long total, int G, int j) {
  return total >= G ? cta_of(bs, total, G) + j : cta_of(bs + j, total, G);
}

#ifdef __CUDACC__
// Prologue of the persistent kernels, run by all `nthreads` threads of the
// CTA: checks the device cu_seqlens against the host sizes `lim`
// (window_valid, every window in every CTA, so all CTAs reach the same
// verdict), scans the per-window iteration counts (each thread sums a
// contiguous run of windows; warp shuffles and a shared array of warp totals
// turn the run sums into prefixes), finds the window holding this CTA's first
// iteration, and lets the first CTA of each schedule row store that row's
// prefix array for the merge kernels (win_prefix_out[row * (batch + 1) + b]).
// Returns false, the same in every thread, when some window is inconsistent;
// then nothing has been written and the caller must return before it loads
// or stores anything.  Otherwise the results land in *total (the row's
// iterations), *b0 and *pre_b0 (shared memory) after the closing
// __syncthreads.  `warp_tot` needs one slot per warp.
template <bool ROW>
__device__ inline bool plan_schedule(const int32_t* cu_p, const int32_t* cu_c, int batch, int hkv,
                                     const Tiling& tl, const SeqLimits& lim,
                                     long long* win_prefix_out, long long* warp_tot,
                                     long long* total, int* b0, long long* pre_b0) {
  const int t = threadIdx.x, nt = blockDim.x;
  const int lane = t & 31, warp = t >> 5, nwarps = nt >> 5;
  const int per = ceil_div(batch, nt);
  const int w0 = t * per;
  const int w1 = (w0 + per < batch) ? w0 + per : batch;
  const int rg = ROW ? row_grid(tl) : tl.grid;
  const int row = ROW ? (int)blockIdx.x / rg : 0, j = ROW ? (int)blockIdx.x % rg : (int)blockIdx.x;
  auto work = [&](int b) {
    const int lp = cu_p[b + 1] - cu_p[b], lc = cu_c[b + 1] - cu_c[b];
    return (long long)hkv * (ROW ? head_work_row(tl, lp, lc, row) : head_work(tl, lp, lc));
  };
  bool bad = false;
  for (int b = w0; b < w1; ++b) bad |= !window_valid(cu_p, cu_c, b, batch, lim);
  if (__syncthreads_or(bad)) return false;
  long long sum = 0;
  for (int b = w0; b < w1; ++b) sum += work(b);
  long long inc = sum;  // inclusive scan within the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += v;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  long long base = 0, all = 0;
  for (int w = 0; w < nwarps; ++w) {
    const long long v = warp_tot[w];
    if (w < warp) base += v;
    all += v;
  }
  long long run = base + inc - sum;  // exclusive prefix of window w0
  const long long start = cta_begin(j, all, rg);
  long long* wp_row = win_prefix_out + (size_t)row * (batch + 1);
  for (int b = w0; b < w1; ++b) {
    const long long wb = work(b);
    if (j == 0) wp_row[b] = run;
    if (wb > 0 && run <= start && start < run + wb) {
      *b0 = b;
      *pre_b0 = run;
    }
    run += wb;
  }
  if (t == 0) {
    *total = all;
    if (j == 0) wp_row[batch] = all;
  }
  __syncthreads();
  return true;
}

#endif  // __CUDACC__

}  // namespace cfa
