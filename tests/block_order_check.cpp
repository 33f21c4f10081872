// Host check of the causal kernels' block order (grouped_rank_order,
// order_head_group in block_order.h): for every grid of nblk x BH blocks
// and every head-group size, the linear block indices map one-to-one onto
// (rank, head) pairs, ranks run heaviest-first within a group, and a group
// holds at most g heads.  Prints "ok" and exits 0 when every case holds.
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
  std::printf("%d grids ok\n", cases);
  return 0;
}
