// Work decomposition shared by the host planner and the kernels.
//
// Query rows are packed GQA-style: a query tile holds `tpt` consecutive chunk
// tokens times the g = Hq/Hkv query heads that read one KV head, row
// r = token_local * g + head_local (rows = tpt * g <= 128).  Every row of a
// tile therefore reads the same K/V tiles, and the causal edge of a tile spans
// only tpt tokens.
//
// The keys of a window are walked as one list of 128-row tiles: the ceil(Lp /
// 128) prefix tiles first, then the chunk tiles that some row of the query
// block can see (chunk key j is visible to token t iff j <= t; the prefix is
// fully visible).  A query block's list is cut into splits of
// `tiles_per_split` tiles; each split is one CTA, and its partial (O, LSE) or
// dQ is merged afterwards when a block has more than one split.
#pragma once

#include <stdint.h>

namespace cfa {

constexpr int kTileM = 128;  // query rows per tile (TMEM lanes)
constexpr int kTileN = 128;  // keys per tile

struct Tiling {
  int g;                // query heads per KV head
  int tpt;              // chunk tokens per query tile
  int rows;             // valid rows per query tile = tpt * g
  int q_per_cta;        // query tiles per CTA (a query block)
  int tiles_per_split;  // key tiles per split
  int n_qblk_max;       // query blocks per window, upper bound
  int n_split_max;      // splits per query block, upper bound
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Key tiles seen by a query block whose first token is t0 and which spans
// `tok_blk` tokens, in a window with lp prefix rows and lc chunk rows.
__host__ __device__ inline int block_key_tiles(int lp, int lc, int t0, int tok_blk) {
  const int t_hi = (t0 + tok_blk < lc) ? (t0 + tok_blk) : lc;
  return ceil_div(lp, kTileN) + ceil_div(t_hi, kTileN);
}

__host__ __device__ inline int block_splits(const Tiling& tl, int lp, int lc, int qblk) {
  const int tok_blk = tl.q_per_cta * tl.tpt;
  return ceil_div(block_key_tiles(lp, lc, qblk * tok_blk, tok_blk), tl.tiles_per_split);
}

}  // namespace cfa
