// Stream-K helpers shared by the FP32 SIMT kernel and the CTA-pair
// tensor-core kernel.  A stream-K launch lays the K-steps ("units") of the
// tiles past the last whole wave end to end, tile by tile, and gives worker
// c (a CTA, or a CTA pair) the contiguous units [sk_begin(c), sk_begin(c+1)).
// Each worker's range is at most one tile long, so it ends in the tile it
// starts in or in the next one.  Workers that do not finish a tile leave
// their partial sum in a workspace and raise flags; the tile's finisher adds
// the parts in worker order.
#ifndef G3_STREAM_K_CUH
#define G3_STREAM_K_CUH

#include <cstdint>

namespace g3 {

__host__ __device__ __forceinline__ long long sk_begin(long long c, long long units, int workers) {
  return c * units / workers;
}

// The workers whose ranges meet the units [T0, T1) of one tile (cfirst ..
// clast) and its finisher: the worker whose share of the tile ends latest
// within its own range (the first on a tie), so its wait is the shortest.
// Only finishers wait, and only on workers with a lower index or on the
// first piece of a range (which no wait precedes), so the waits form no
// cycle.
__host__ __device__ __forceinline__ void sk_tile_workers(long long T0, long long T1, long long U,
                                                         int G, int* cfirst, int* clast, int* fin) {
  const int c0 = (int)(((T0 + 1) * G + U - 1) / U) - 1;
  const int c1 = (int)((T1 * G + U - 1) / U) - 1;
  int f = c0;
  long long best = -1;
  for (int c = c0; c <= c1; ++c) {
    const long long b = sk_begin(c, U, G);
    const long long e = sk_begin(c + 1, U, G) < T1 ? sk_begin(c + 1, U, G) : T1;
    if (e - b > best) {
      best = e - b;
      f = c;
    }
  }
  *cfirst = c0;
  *clast = c1;
  *fin = f;
}

// The most workers that meet in one of `tiles` tiles of `units_per_tile`
// units each, spread over G workers.
__host__ __device__ __forceinline__ int sk_max_share(long long tiles, int units_per_tile, int G) {
  const long long U = tiles * units_per_tile;
  int share = 1;
  for (long long t = 0; t < tiles; ++t) {
    int c0, c1, f;
    sk_tile_workers(t * units_per_tile, (t + 1) * units_per_tile, U, G, &c0, &c1, &f);
    if (c1 - c0 + 1 > share) share = c1 - c0 + 1;
  }
  return share;
}

#ifdef __CUDACC__
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
#endif

}  // namespace g3

#endif  // G3_STREAM_K_CUH
