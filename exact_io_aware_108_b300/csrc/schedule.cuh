// schedule.cuh -- which work item each CTA of the attention kernels takes,
// and which rows of the backward's workspace it touches. Plain integer
// arithmetic, callable from host code too, so the same functions the kernels
// run can be checked exhaustively on the CPU (every work item taken exactly
// once, every index inside its buffer) for any launch shape.
#pragma once

namespace fa {

struct WorkItem {
  int bh;    // [B*H] (forward) or [B*Hkv] (backward) head index
  int tile;  // query-tile pair (two-tile forward), query tile, or key tile
};

// Grouped, heaviest-first launch order: CTAs are taken in groups of `hgroup`
// heads (the last group may be smaller); inside a group the tile index runs
// slowest, so the CTAs of equal tile index of the group's heads start
// together. Two-tile forward: tiles = query-tile pairs (reversed for causal
// attention: the last pairs see the most key tiles). Backward: tiles = key
// tiles (causal: the first key tiles see the most query tiles).
__host__ __device__ inline WorkItem grouped_item(int block, int n_heads, int n_tiles, int hgroup,
                                                 bool reverse) {
  const int grp = block / (hgroup * n_tiles);
  const int rem = block - grp * hgroup * n_tiles;
  const int nh = hgroup < n_heads - grp * hgroup ? hgroup : n_heads - grp * hgroup;
  WorkItem w;
  w.tile = rem / nh;
  w.bh = grp * hgroup + rem % nh;
  if (reverse) w.tile = n_tiles - 1 - w.tile;
  return w;
}

// One query tile per CTA, heads contiguous in the grid (reversed tile order
// for causal attention).
__host__ __device__ inline WorkItem tile_item(int block, int nqt, bool reverse) {
  WorkItem w;
  w.bh = block / nqt;
  w.tile = block % nqt;
  if (reverse) w.tile = nqt - 1 - w.tile;
  return w;
}

// Split-KV: share `split` of `splits` takes the contiguous key tiles
// [*lo, *lo + *n) of a row's n_all tiles.
__host__ __device__ inline void split_share(int n_all, int split, int splits, int *lo, int *n) {
  *lo = static_cast<int>(static_cast<long long>(n_all) * split / splits);
  *n = static_cast<int>(static_cast<long long>(n_all) * (split + 1) / splits) - *lo;
}

// [B*Hkv] key/value head read by query head bh ([B*H] index).
__host__ __device__ inline int kv_head_of(int bh, int H, int Hkv) {
  return (bh / H) * Hkv + (bh % H) / (H / Hkv);
}

// [B*H] index of query head g of the group that reads key/value head bkv.
__host__ __device__ inline int q_head_of(int bkv, int g, int H, int Hkv) {
  return (bkv / Hkv) * H + (bkv % Hkv) * (H / Hkv) + g;
}

}  // namespace fa
