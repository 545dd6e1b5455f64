// Reads stream-K queries from stdin and prints the partition that the
// kernels compute with csrc/stream_k.cuh, so that a CPU test can check it:
//   tiles units_per_tile workers
// -> for each tile "cfirst clast finisher", then "share <max workers per tile>".
// The header's host/device qualifiers are defined away for the host compiler.
#define __host__
#define __device__
#define __forceinline__ inline
#include <cstdio>

#include "stream_k.cuh"

int main() {
  long long tiles;
  int upt, G;
  while (std::scanf("%lld %d %d", &tiles, &upt, &G) == 3) {
    const long long U = tiles * upt;
    for (long long t = 0; t < tiles; ++t) {
      int c0, c1, f;
      g3::sk_tile_workers(t * upt, (t + 1) * upt, U, G, &c0, &c1, &f);
      std::printf("%d %d %d\n", c0, c1, f);
    }
    std::printf("share %d\n", g3::sk_max_share(tiles, upt, G));
  }
  return 0;
}
