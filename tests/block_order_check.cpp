// Host check of the block-order helpers in block_order.h:
//  - grouped_rank_order / order_head_group (the causal kernels' order): for
//    every grid of nblk x BH blocks and every head-group size, the linear block
//    indices map one-to-one onto (rank, head) pairs, ranks run heaviest-first
//    within a group, and a group holds at most g heads;
//  - tail_split_items / split_block_item / bwd_tail_split_items (the
//    backward's split last wave):
//    the split items are exactly the last partial wave when it is at most half
//    the SMs, and the grid's blocks cover every unsplit item once and both
//    halves of every split item.
// Prints "ok" and exits 0 when every case holds.
#include <cstdio>
#include <vector>

#include "block_order.h"

int main() {
  int cases = 0;
  for (int nblk = 1; nblk <= 40; nblk += 3) {
    for (int BH = 1; BH <= 37; BH += 2) {
      for (int g = 1; g <= BH + 2; ++g) {
        const int gg = g > BH ? BH : g;  // order_head_group never returns more than BH
        std::vector<int> seen(static_cast<size_t>(nblk) * BH, 0);
        int prev_grp_first_head = -1, prev_rank = -1, prev_grp = -1;
        for (int L = 0; L < nblk * BH; ++L) {
          int rank = -1, bh = -1;
          attn::grouped_rank_order(L, nblk, BH, gg, rank, bh);
          if (rank < 0 || rank >= nblk || bh < 0 || bh >= BH) {
            std::printf("out of range: nblk=%d BH=%d g=%d L=%d -> rank=%d bh=%d\n", nblk, BH, gg, L, rank, bh);
            return 1;
          }
          if (seen[static_cast<size_t>(bh) * nblk + rank]++) {
            std::printf("duplicate: nblk=%d BH=%d g=%d L=%d\n", nblk, BH, gg, L);
            return 1;
          }
          const int grp = bh / gg;
          if (grp < prev_grp || (grp == prev_grp && rank < prev_rank)) {  // ranks never go back within a group
            std::printf("order: nblk=%d BH=%d g=%d L=%d\n", nblk, BH, gg, L);
            return 1;
          }
          if (grp != prev_grp) prev_grp_first_head = grp * gg;
          if (bh < prev_grp_first_head || bh >= prev_grp_first_head + gg) {
            std::printf("group: nblk=%d BH=%d g=%d L=%d\n", nblk, BH, gg, L);
            return 1;
          }
          prev_grp = grp;
          prev_rank = rank;
        }
        ++cases;
      }
    }
  }
  // group size: budget / bytes, clamped to [1, BH]
  if (attn::order_head_group(32, int64_t{4} << 20, int64_t{32} << 20) != 8 ||
      attn::order_head_group(32, int64_t{1} << 30, int64_t{32} << 20) != 1 ||
      attn::order_head_group(4, 1, int64_t{32} << 20) != 4) {
    std::printf("order_head_group\n");
    return 1;
  }
  // tail split: which items of a grid's last partial wave run as two halves
  for (int S : {1, 7, 148, 152}) {
    for (int64_t W = 1; W <= 3000; W += (W < 400 ? 1 : 7)) {
      const int r = attn::tail_split_items(W, S);
      const int64_t rem = W % S;
      if (r > 0) {
        if (r != rem || 2 * r > S || (W - r) % S != 0) {
          std::printf("tail split: W=%lld S=%d r=%d\n", static_cast<long long>(W), S, r);
          return 1;
        }
      } else if (rem != 0 && 2 * rem <= S) {
        std::printf("tail split missed: W=%lld S=%d\n", static_cast<long long>(W), S);
        return 1;
      }
      // blocks -> (item, half): unsplit items once, split items once per half
      const int split_from = static_cast<int>(W - r);
      std::vector<int> whole(static_cast<size_t>(W), 0), halves(static_cast<size_t>(W), 0);
      for (int b = 0; b < W + r; ++b) {
        int item = -1, half = -2, pair = -1;
        attn::split_block_item(b, split_from, item, half, pair);
        if (item < 0 || item >= W || (half == -1) != (item < split_from) || half < -1 || half > 1 ||
            pair != (half < 0 ? 0 : item - split_from)) {
          std::printf("split mapping: W=%lld r=%d b=%d -> item=%d half=%d\n", static_cast<long long>(W), r, b,
                      item, half);
          return 1;
        }
        if (half < 0) ++whole[static_cast<size_t>(item)];
        else halves[static_cast<size_t>(item)] |= 1 << half;
      }
      for (int64_t i = 0; i < W; ++i) {
        const bool ok = i < split_from ? (whole[static_cast<size_t>(i)] == 1 && halves[static_cast<size_t>(i)] == 0)
                                       : (whole[static_cast<size_t>(i)] == 0 && halves[static_cast<size_t>(i)] == 3);
        if (!ok) {
          std::printf("split coverage: W=%lld r=%d item=%lld\n", static_cast<long long>(W), r,
                      static_cast<long long>(i));
          return 1;
        }
      }
      ++cases;
    }
  }
  // the backward's policy: never under the causal mask or for a single query
  // tile; otherwise the generic rule over ceil(N / 128) * BH items
  for (int S : {148, 152}) {
    for (int BH = 1; BH <= 40; BH += 3) {
      for (int N : {1, 128, 129, 1000, 8192, 32768}) {
        const int ntq = (N + 127) / 128;
        const int want = ntq < 2 ? 0 : attn::tail_split_items(static_cast<int64_t>(ntq) * BH, S);
        if (attn::bwd_tail_split_items(BH, N, 1, S) != 0 || attn::bwd_tail_split_items(BH, N, 0, S) != want) {
          std::printf("bwd tail split: BH=%d N=%d S=%d\n", BH, N, S);
          return 1;
        }
        ++cases;
      }
    }
  }
  std::printf("%d grids ok\n", cases);
  return 0;
}
