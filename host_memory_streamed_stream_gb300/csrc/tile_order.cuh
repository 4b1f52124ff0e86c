// Block order of the causal attention grids.
//
// Under a causal mask the work of a 128-row tile grows (query tiles) or shrinks (key tiles)
// linearly with its index. With the grid laid out head by head, the last head's heaviest tile
// is handed out near the end and keeps one SM busy while the others idle: at the 7B shapes
// (64 heads x 32 tiles, 152 SMs) that tail costs about 8 % of the dK/dV kernel and 15 % of the
// forward; at the 14B GQA shapes (8 KV heads x 32 tiles) about 40 % of the dK/dV kernel.
//
// The grids are therefore one-dimensional and blocks are handed out heaviest tile first over
// groups of kHeadGroup (head, batch) pairs: block i of a group takes tile rank i / g of head
// pair i % g (g = the group's size). The heavy tiles of a group start first and its light
// tiles fill the tail, while the CTAs running at one time read the operands of at most a few
// groups, which stay in L2.
#pragma once

namespace mt {

constexpr int kHeadGroup = 16;

struct TileSlot {
  int rank;  // 0 = the heaviest tile of its head
  int hb;    // head + n_heads * batch
};

// Slot of block `lin` in a grid of n_tiles x n_hb blocks.
__host__ __device__ inline TileSlot heavy_first_slot(int lin, int n_tiles, int n_hb) {
  const int per_group = n_tiles * kHeadGroup;
  const int g = lin / per_group;
  const int within = lin - g * per_group;
  const int gsz = (n_hb - g * kHeadGroup) < kHeadGroup ? (n_hb - g * kHeadGroup) : kHeadGroup;
  return {within / gsz, g * kHeadGroup + within % gsz};
}

}  // namespace mt
