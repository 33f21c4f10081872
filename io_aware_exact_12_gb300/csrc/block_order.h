// block_order.h -- the order in which the causal kernels visit their blocks
// (host and device; no other dependencies, so host tests can include it).
#pragma once

#include <stdint.h>

#ifndef __CUDACC__
#ifndef __host__
#define __host__
#endif
#ifndef __device__
#define __device__
#endif
#endif

namespace attn {

// Block order of the causal kernels.  Under the causal mask a block's work
// grows with its distance from the diagonal; issued head after head, the
// heaviest blocks of the last heads would start last and leave SMs idle at the
// end.  Linear block index L (blockIdx.x fastest) is mapped instead so that
// within each group of g heads every head's heaviest block comes first, then
// every head's next-heaviest, and so on: rank 0 is the heaviest block of its
// head.  g keeps the operands of the heads in flight a small part of L2.
__host__ __device__ inline void grouped_rank_order(int L, int nblk, int BH, int g, int& rank, int& bh) {
  const int grp = L / (g * nblk);
  const int rem = L - grp * g * nblk;
  const int gl = (BH - grp * g < g) ? BH - grp * g : g;  // heads in this (possibly last, short) group
  rank = rem / gl;
  bh = grp * g + (rem - rank * gl);
}

// Heads per group for grouped_rank_order: as many as keep `bytes_per_head`
// of streamed operands within `budget` bytes, at least one.  The forward
// (read-only K/V) measured best with the group as large as L2 (128 MB), the
// backward (dQ reductions into the same lines) with 32 MB.
inline int order_head_group(int BH, int64_t bytes_per_head, int64_t budget) {
  int64_t g = bytes_per_head > 0 ? budget / bytes_per_head : BH;
  if (g < 1) g = 1;
  if (g > BH) g = BH;
  return static_cast<int>(g);
}

// Split of a grid's last partial wave.  W equal-cost items on S SMs run as
// W / S full waves plus a last wave of r = W mod S items while S - r SMs idle;
// when 2 r <= S, those r items can each run as two blocks over half of the
// item's range, so the last wave takes half as long.  Returns how many items
// to split (0: none).
__host__ __device__ inline int tail_split_items(int64_t W, int S) {
  if (W <= 0 || S <= 0) return 0;
  const int64_t r = W % S;
  return (r > 0 && 2 * r <= S) ? static_cast<int>(r) : 0;
}

// The backward's use of it: without the causal mask every (key tile, head)
// item costs the same, so the ceil(N/128) * BH items on `sms` SMs may end with
// a short wave; a key tile with a single query tile has nothing to split.
__host__ __device__ inline int bwd_tail_split_items(int BH, int N, int causal, int sms) {
  if (causal) return 0;
  const int64_t ntq = (static_cast<int64_t>(N) + 127) / 128;
  if (ntq < 2) return 0;
  return tail_split_items(ntq * BH, sms);
}

// Block b of a grid of W + r blocks whose last r items are split (split_from =
// W - r): the item it works on, which half of the item's range (-1: all) and,
// for a split item, its pair index item - split_from.  Blocks below
// split_from map one to one; from there on, blocks come in pairs (half 0,
// half 1) of consecutive items.
__host__ __device__ inline void split_block_item(int b, int split_from, int& item, int& half, int& pair) {
  item = b;
  half = -1;
  pair = 0;  // index of the split pair (0 for blocks below split_from)
  if (b >= split_from) {
    pair = (b - split_from) >> 1;
    half = (b - split_from) & 1;
    item = split_from + pair;
  }
}

}  // namespace attn
