// Launch planning: the wave models that pick a kernel configuration from the
// problem shape and the GPU's SM count.  Plain host arithmetic with no CUDA
// types, so that the library and a CPU test compile the same code.
//
// Every model counts waves ("Kernel 性能从何而来", "SM 占用率与资源压力": the CTA
// slots, registers and shared memory of an SM bound how many CTAs run at
// once, so tiles run in waves and a partial last wave leaves SMs idle).
// Per-column and per-tile costs are measured on GB300.
#pragma once

namespace g3 {
namespace plan {

// Tile width of the single-CTA tensor-core kernel: every wave of 128 x bn
// tiles costs about one tile-time, so minimise waves(bn) * bn * cost(bn).
// Relative per-column costs at 8192^3, where the last-wave loss is small:
// 1.000 (256), 1.012 (192), 1.070 (128); 224-wide MMAs cost 1.115 and are
// never chosen automatically.  Ties go to the wider tile.
inline int tc_bn(int M, int N, int num_sms) {
  static const int cands[] = {256, 192, 128};
  static const int cost_milli[] = {1000, 1012, 1070};
  const long long tiles_m = (M + 127) / 128;
  int best = 256;
  long long best_cost = -1;
  for (int i = 0; i < 3; ++i) {
    const int bn = cands[i];
    const long long tiles = tiles_m * ((N + bn - 1) / bn);
    const long long waves = (tiles + num_sms - 1) / num_sms;
    const long long cost = waves * bn * cost_milli[i];
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// Single CTA (pair = 1) or CTA pair (pair = 2), and the tile width: the same
// wave model over both families.  A pair tile (256 x bn) runs on two SMs, so
// per SM it is a 128 x bn tile; its per-column cost at 8192^3 is 0.882
// (bn = 256) and 1.018 (bn = 128) of the single-CTA 256-wide tile.  A
// partial last wave of 256-wide pair tiles that fits in half the pairs runs
// as 128-wide halves when `split_allowed`, so it costs one 128-wide wave.  On
// a tie the 128-wide pair kernel, evaluated first, is kept.
inline void tc_config(int M, int N, int num_sms, bool split_allowed, int* pair, int* bn) {
  *pair = 1;
  *bn = tc_bn(M, N, num_sms);
  const long long single_tiles = (long long)((M + 127) / 128) * ((N + *bn - 1) / *bn);
  const long long single_waves = (single_tiles + num_sms - 1) / num_sms;
  const int single_cost_milli = *bn == 256 ? 1000 : *bn == 192 ? 1012 : 1070;
  long long best = single_waves * *bn * single_cost_milli;
  static const int pair_bn[] = {128, 256};
  static const int pair_cost_milli[] = {1018, 882};
  const int clusters = num_sms / 2 > 0 ? num_sms / 2 : 1;
  for (int i = 0; i < 2; ++i) {
    const long long tiles = (long long)((M + 255) / 256) * ((N + pair_bn[i] - 1) / pair_bn[i]);
    const long long rem = tiles % clusters;
    const long long wave = (long long)pair_bn[i] * pair_cost_milli[i];
    const bool halved = pair_bn[i] == 256 && split_allowed && rem > 0 && 2 * rem <= clusters;
    const long long cost =
        (tiles / clusters) * wave + (rem == 0 ? 0 : halved ? 128LL * pair_cost_milli[0] : wave);
    if (cost < best) {
      best = cost;
      *pair = 2;
      *bn = pair_bn[i];
    }
  }
}

// CTA-pair kernel, 256-wide tiles, `rem` tiles past the last whole wave of
// `pairs`: the pairs of a stream-K tail, min(pairs, K-steps / 8), so that
// each pair streams at least 8 K-steps; 0 (no stream-K) when a tile has
// fewer than 8 K-steps, since then a pair's range could span three tiles.
constexpr int kTcSkMinSteps = 8;
inline int tc_sk_pairs(long long rem, int k_tiles, int pairs) {
  if (rem <= 0 || pairs <= 0 || k_tiles < kTcSkMinSteps) return 0;
  const long long by_work = rem * k_tiles / kTcSkMinSteps;
  const long long g = by_work < pairs ? by_work : pairs;
  return g < rem ? 0 : (int)g;
}

// How those `rem` tiles run, in tile-times: whole tiles (0) cost one;
// half-width tiles (1, when 2 rem <= pairs) cost kTcHalfTile; stream-K over
// sk_pairs pairs (2) costs rem / sk_pairs of a tile plus kTcSkExchange for
// writing, waiting for and adding the partial tiles.  Measured on GB300 the
// exchange costs more than a whole tile: each finisher warp adds the other
// pairs' parts to its accumulator chunk by chunk after its own piece, and
// that fix-up (15-30 us) is on the critical path (bf16 4096^3: 78.5 us with
// half-width tiles, 84.6 whole, 101.0 stream-K; 2048 x 4096 x 4096: 47.8
// whole, 64.1 stream-K; 8192^3: 578 half, 595 stream-K), so the model
// never picks it; gemm_force_split_tiles(2) still runs it.
constexpr double kTcHalfTile = 0.58;
constexpr double kTcSkExchange = 1.0;
inline int tc_tail(long long rem, int pairs, bool half_ok, int sk_pairs) {
  if (rem <= 0 || pairs <= 0) return 0;
  int best = 0;
  double t = 1.0;
  if (half_ok && kTcHalfTile < t) {
    best = 1;
    t = kTcHalfTile;
  }
  if (sk_pairs > 0 && (double)rem / sk_pairs + kTcSkExchange < t) best = 2;
  return best;
}

// Time of `units` CTAs, each `unit` of a whole tile, with `slots` resident at
// once, in tiles run two to an SM; a round of at most one CTA per SM runs
// about 1.9x as fast (FP32 SIMT kernel on GB300, 4096^3 slices: 304 tiles two
// to an SM take 679 us, 16 tiles alone 361 us).
inline double rounds_time(long long units, double unit, long long slots, int sms) {
  const long long rest = units % slots;
  return unit * (double)(units / slots) + (rest == 0 ? 0.0 : rest <= sms ? 0.53 * unit : unit);
}

// FP32 SIMT kernel (two CTAs per SM): whether the tiles past the last whole
// wave run as a second launch with K split over clusters of `split` CTAs.
// `max_clusters` is how many such clusters are resident at once; each rank
// needs at least `min_k_tiles` K-slices.  The quarter-tiles must finish the
// partial wave sooner by more than a tenth of a tile (the reduction and the
// shorter pipelines).
inline bool simt_split(long long tiles, int k_tiles, int num_sms, int max_clusters, int split,
                       int min_k_tiles, bool split_allowed) {
  const long long slots = 2LL * num_sms;
  const long long rest = tiles % slots;
  if (!split_allowed || rest == 0 || k_tiles < split * min_k_tiles || max_clusters <= 0)
    return false;
  const long long split_slots = (long long)split * max_clusters;
  return rounds_time(rest * split, 1.0 / split, split_slots, num_sms) + 0.1 <
         rounds_time(rest, 1.0, slots, num_sms);
}

// FP32 SIMT kernel: one candidate configuration and its estimated time.
// `time` is in units of one 128 x 128 x K tile computed by a whole SM at the
// narrow kernel's rate; `split` is 1 (whole tiles only), 4 (narrow: clusters
// of four CTAs share the K range of each tile past the last whole wave) or
// 0 (wide: those tiles' K-slices are split evenly over the SMs, stream-K).
struct SimtOption {
  double time = 1e300;
  int split = 1;
};

// Per-SM rate of the wide configuration (8 x 16 register tiles, 128 x 256 C
// tiles, one CTA per SM) relative to the narrow one (8 x 8, 128 x 128, two
// CTAs per SM): the bare inner loops retire 0.816 and 0.759 of the FP32 peak
// on one GB300.
constexpr double kSimtWideRate = 1.075;
// The wide configuration is chosen only when its estimate is below this
// fraction of the narrow one (the estimates' error at short K: 2560 x 2048 x
// 1024 modelled 4 % faster on wide tiles, measured 7 % slower).
constexpr double kSimtWideMargin = 0.97;

// The estimate for register-tile width `tn` (8: narrow, 16: wide) with
// `tiles` C tiles of that configuration.  max_clusters2/4: clusters of 2 and
// of 4 CTAs of its split kernel resident at once (0: none, or not queried);
// each rank needs at least `min_k_tiles` K-slices.
//   narrow: a wave is two tiles per SM; the partial last wave either runs
//           whole (rounds_time: about 0.53 of a wave when it is at most one
//           CTA per SM) or K-split over clusters of four, as simt_split
//           decides (its tenth-of-a-tile margin is part of the decision, not
//           of the estimate);
//   wide:   a wave is one tile per SM and a partial round costs a whole one;
//           the partial last wave either runs whole or stream-K: its
//           K-slices spread over min(SMs, slices / (2 x 8)) CTAs, one per SM
//           (rest / CTAs of a wave), plus 0.02 of a tile for the partial sums'
//           exchange; stream-K needs at least 16 K-slices a tile, so that no
//           CTA's range is longer than a tile.
// Measured on one GB300 (K = 4096, in narrow waves of 0.699 ms): 4096^3
// 3.35 narrow split / 3.19 wide stream-K (estimates 3.38 / 3.15); 2048^2
// 0.866 / 0.851 (0.88 / 0.80); 8192^2 13.3 / 12.6 (13.5 / 12.6).
inline SimtOption simt_option(int tn, long long tiles, int k_tiles, int num_sms, int max_clusters2,
                              int max_clusters4, int min_k_tiles, bool split_allowed) {
  SimtOption o;
  if (tiles <= 0 || num_sms <= 0) {
    o.time = 0.0;
    return o;
  }
  if (tn == 8) {
    const long long slots = 2LL * num_sms;
    const double wave = 2.0;  // two tiles per SM
    if (simt_split(tiles, k_tiles, num_sms, max_clusters4, 4, min_k_tiles, split_allowed)) {
      const long long rest = tiles % slots;
      o.split = 4;
      o.time = wave * ((double)(tiles / slots) +
                       rounds_time(rest * 4, 0.25, 4LL * max_clusters4, num_sms));
    } else {
      o.time = wave * rounds_time(tiles, 1.0, slots, num_sms);
    }
    return o;
  }
  (void)max_clusters2;
  (void)max_clusters4;
  const long long slots = num_sms;
  const double wave = 2.0 / kSimtWideRate;  // one 128 x 256 tile per SM
  const long long whole = tiles / slots, rest = tiles % slots;
  o.time = wave * (double)(whole + (rest > 0 ? 1 : 0));
  if (!split_allowed || rest == 0 || k_tiles < min_k_tiles) return o;
  long long ctas = rest * k_tiles / min_k_tiles;
  if (ctas > slots) ctas = slots;
  const double t = wave * ((double)whole + (double)rest / (double)ctas + 0.02);
  if (t < o.time) {
    o.time = t;
    o.split = 0;
  }
  return o;
}

// Decode kernels: CTAs of a cluster that share one column slab's K range.  The
// largest power of two up to `max_split` whose grid still fits two CTAs per
// SM, and no more than the K units there are; `forced` (1, 2, 4 or 8)
// overrides the first choice.
inline int cluster_split(int tiles_n, int k_units, int num_sms, int forced, int max_split) {
  int s = 1;
  if (forced == 1 || forced == 2 || forced == 4 || forced == 8) {
    s = forced;
  } else {
    const int target = 2 * num_sms;
    while (s * 2 <= max_split && tiles_n * s * 2 <= target) s *= 2;
  }
  while (s > 1 && s > k_units) s /= 2;
  return s;
}

}  // namespace plan
}  // namespace g3
