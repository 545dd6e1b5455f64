// Reads planning queries from stdin, one per line, and prints each answer on
// its own line, so that a CPU test can check the library's launch planning
// (csrc/plan.h) without a GPU:
//   tc M N sms split_allowed                    -> "pair bn"
//   bn M N sms                                  -> "bn"
//   simt tiles k_tiles sms max_clusters split min_k_tiles split_allowed -> 0 or 1
//   cluster tiles_n k_units sms forced max_split -> split
//   simtopt tn tiles k_tiles sms clusters2 clusters4 min_k_tiles split_allowed -> "time split"
//   tcsk rem k_tiles pairs                       -> stream-K pairs
//   tctail rem pairs half_ok sk_pairs            -> 0 whole, 1 half-width, 2 stream-K
#include <cstdio>
#include <cstring>

#include "plan.h"

int main() {
  char op[16];
  while (std::scanf("%15s", op) == 1) {
    if (!std::strcmp(op, "tc")) {
      int M, N, sms, allowed, pair = 0, bn = 0;
      if (std::scanf("%d %d %d %d", &M, &N, &sms, &allowed) != 4) return 2;
      g3::plan::tc_config(M, N, sms, allowed != 0, &pair, &bn);
      std::printf("%d %d\n", pair, bn);
    } else if (!std::strcmp(op, "bn")) {
      int M, N, sms;
      if (std::scanf("%d %d %d", &M, &N, &sms) != 3) return 2;
      std::printf("%d\n", g3::plan::tc_bn(M, N, sms));
    } else if (!std::strcmp(op, "simt")) {
      long long tiles;
      int k_tiles, sms, clusters, split, min_k, allowed;
      if (std::scanf("%lld %d %d %d %d %d %d", &tiles, &k_tiles, &sms, &clusters, &split, &min_k,
                     &allowed) != 7)
        return 2;
      std::printf("%d\n",
                  g3::plan::simt_split(tiles, k_tiles, sms, clusters, split, min_k, allowed != 0) ? 1 : 0);
    } else if (!std::strcmp(op, "simtopt")) {
      long long tiles;
      int tn, k_tiles, sms, c2, c4, min_k, allowed;
      if (std::scanf("%d %lld %d %d %d %d %d %d", &tn, &tiles, &k_tiles, &sms, &c2, &c4, &min_k,
                     &allowed) != 8)
        return 2;
      const g3::plan::SimtOption o =
          g3::plan::simt_option(tn, tiles, k_tiles, sms, c2, c4, min_k, allowed != 0);
      std::printf("%.4f %d\n", o.time, o.split);
    } else if (!std::strcmp(op, "tcsk")) {
      long long rem;
      int k_tiles, pairs;
      if (std::scanf("%lld %d %d", &rem, &k_tiles, &pairs) != 3) return 2;
      std::printf("%d\n", g3::plan::tc_sk_pairs(rem, k_tiles, pairs));
    } else if (!std::strcmp(op, "tctail")) {
      long long rem;
      int pairs, half_ok, sk;
      if (std::scanf("%lld %d %d %d", &rem, &pairs, &half_ok, &sk) != 4) return 2;
      std::printf("%d\n", g3::plan::tc_tail(rem, pairs, half_ok != 0, sk));
    } else if (!std::strcmp(op, "cluster")) {
      int tiles_n, k_units, sms, forced, max_split;
      if (std::scanf("%d %d %d %d %d", &tiles_n, &k_units, &sms, &forced, &max_split) != 5) return 2;
      std::printf("%d\n", g3::plan::cluster_split(tiles_n, k_units, sms, forced, max_split));
    } else {
      return 3;
    }
  }
  return 0;
}
