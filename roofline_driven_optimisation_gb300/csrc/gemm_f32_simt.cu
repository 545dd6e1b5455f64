// FP32 SGEMM on the CUDA cores: C = alpha*A*B + beta*C, row-major fp32.
//
// FP32 has no dense tensor-core route, so this path is the three-level tiling
// of "CUDA 算子工程 ch.10 朴素 GEMM 与 Roofline 分析", section 10.4, done with
// FFMA instead of MMA:
//   * block tile 128 x BN, K-slices of 16 (section 10.4.1: each K column of
//     the A and B tiles feeds 128 x BN FMAs);
//   * warp tile 64 x 4*TN (10.4.1: the warp tile's reuse of shared memory);
//   * register tile 8 x TN per thread (10.4.1: every loaded element is used
//     TN or 8 times; section 10.6 is the 4 x 4 version of the same idea),
//     accumulated with the packed fma.rn.f32x2 (two IEEE fp32 FMAs per
//     instruction).
// Two register tiles share the code:
//   TN = 16: 128 x 256 C tiles, one CTA of eight warps per SM, ~200
//            registers a thread, an 8-stage ring -- the large-shape kernel;
//   TN = 8:  128 x 128 C tiles, two CTAs per SM at 128 registers, 5 stages --
//            for shapes whose tile count the wide tiles cover badly.
// The wide tile is faster because of the register file, not shared memory:
// each packed FMA reads its accumulator pair, one operand pair and one
// operand broadcast from a single register, and the issue order keeps the B
// pair the same over consecutive FMAs (for each B pair, all 8 rows), so only
// the accumulator and the broadcast A value change from one FMA to the next.
// A bare copy of the inner loop (shared-memory fragments and FMAs, no TMA)
// retires 0.78 of the FP32 peak with the old order (for each row, all B
// pairs) and the 8 x 8 tile, 0.80 with this order, and 0.86 with this order
// and the 8 x 16 tile, on one GB300; handing the FMA a full A pair instead of
// a broadcast was slower (0.71).
//
// The K-slices stream through a shared-memory ring filled by TMA ("Kernel
// 性能从何而来", section "优化阶梯": TMA-backed loads are the first big step).
// A slot is handed to the eight warps by an mbarrier that the copy
// completes, and handed back by a counter: the last warp to finish with a
// slot issues its refill, so no warp ever waits for the others to release
// one (same page, "通过重叠执行减少硬件空闲": keep every unit busy).
//
// Shared-memory bank conflicts ("CUDA 算子工程 ch.4 内存层级与代价表", sections
// 4.3.1-4.3.4): the A tile is stored [m][k] (64 bytes per row) with the TMA
// 64-byte swizzle, so the eight rows a warp reads with one 64-bit load land
// on eight disjoint groups of banks; B is read along n, where a warp needs
// only 64 contiguous bytes per load.  TMA zero-fills outside the matrix, so
// ragged M, N, K need no guards in the main loop (the role the bounds checks
// play in the thread-tile kernel of ch.10, 10.6).
//
// Waves ("Kernel 性能从何而来", "SM 占用率与资源压力": CTA slots, registers and
// shared memory bound the CTAs an SM holds): C tiles run in waves of
// CTAs-per-SM x SMs, and a partial last wave leaves SMs idle.  Its tiles can
// instead run as a second launch in which a cluster of SPLIT CTAs shares each
// tile's K range; the partial sums meet in distributed shared memory (no
// global workspace) and are added in rank order, so results stay
// deterministic.  4096^3 on 152 SMs with 128 x 256 tiles: 512 tiles are
// three waves of 152 and 56 tiles, which run as 112 half-K tiles.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "epilogue.cuh"
#include "internal.h"
#include "plan.h"
#include "ptx.cuh"
#include "stream_k.cuh"

namespace g3 {
namespace {

constexpr int BM = kSimtBM, BK = kSimtBK;
constexpr int COMPUTE_WARPS = 8;
constexpr int THREADS = COMPUTE_WARPS * 32;

template <int TN_>
struct SimtCfg {
  static constexpr int TN = TN_;                 // C columns per thread
  static_assert(TN == 8 || TN == 16, "register tiles are 8 x 8 or 8 x 16");
  static constexpr int WN = 4 * TN;              // warp tile width (4 lanes along n)
  static constexpr int BN = 4 * WN;              // four warps along n
  static constexpr int CTAS_PER_SM = TN == 8 ? 2 : 1;
  static constexpr int STAGES = TN == 8 ? 5 : 8;
  static constexpr int A_STAGE_BYTES = BM * BK * 4;
  static constexpr int B_STAGE_BYTES = BK * BN * 4;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int SMEM_BYTES = RING_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  // A split CTA's partial tile, [BM][PART_LD] fp32 over the idle ring: a row
  // pitch of BN + 4 floats puts the eight rows one 128-bit store covers on
  // distinct banks.
  static constexpr int PART_LD = BN + 4;
  static_assert(BM * PART_LD * 4 <= RING_BYTES, "partial tile fits the ring");
  static_assert(STAGES * 8 + 16 + 2 * STAGES * 4 <= 192, "barrier area (the stall barrier sits at 192)");
};
static_assert(SimtCfg<8>::BN == kSimtBN8 && SimtCfg<16>::BN == kSimtBN16, "tile widths");

struct SimtParams {
  GemmArgs a;
  int tiles_m, tiles_n;
  int c_vec;      // C pointer 16-byte aligned and ldc % 4 == 0
  int tile_base;  // raster index of the split launch's first C tile
  // stream-K launch (SPLIT == 0): the tiles from tile_base on, as sk_units
  // K-slices in tile order, split evenly over sk_ctas CTAs
  long long sk_units;
  int sk_ctas;
  float* sk_partials;     // [sk_ctas][kSkMaxSeg][BM][BN] fp32 partial tiles
  unsigned* sk_flags;     // [sk_ctas][kSkMaxSeg][8 warps]: 1 = that warp's part is written
};

// Stream-K: a CTA's K-slice range is at most one tile long, so it touches at
// most two tiles.
constexpr int kSkMaxSeg = 2;

__device__ __forceinline__ float2 lds64(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// Two consecutive float pairs from shared memory as packed 64-bit registers.
__device__ __forceinline__ void lds_pairs(uint32_t addr, uint64_t& p0, uint64_t& p1) {
  asm volatile("ld.shared.v2.b64 {%0,%1}, [%2];" : "=l"(p0), "=l"(p1) : "r"(addr));
}

// (x, x) as a packed pair.
__device__ __forceinline__ uint64_t dup2(float x) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}

// d.lo += a.lo * b.lo; d.hi += a.hi * b.hi -- two IEEE fp32 FMAs in one
// instruction, which halves the FMA issue slots of the outer product.  The
// product is issued as b * a: the B pair, the same over consecutive FMAs,
// takes the first multiplicand slot (on GB300: 8192^2 x 4096 0.725 -> 0.730
// of the FP32 peak on 8 x 8 tiles, unchanged on 8 x 16; an FMA rounds once,
// so the result is the same bits).
__device__ __forceinline__ void ffma2(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %2, %1, %0;" : "+l"(d) : "l"(a), "l"(b));
}

__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Four consecutive C elements of row m from column n on: v holds alpha*A*B;
// adds beta*C, then bias and activation (EPI), and stores what lies inside C.
template <bool EPI>
__device__ __forceinline__ void store_quad(const GemmArgs& a, int c_vec, long long m, long long n,
                                           float v[4]) {
  float* cp = static_cast<float*>(a.C) + m * a.ldc + n;
  const bool beta_nz = a.beta != 0.f;
  if (c_vec && n + 3 < a.N) {
    if (beta_nz) {
      const float4 c = *reinterpret_cast<const float4*>(cp);
      v[0] = fmaf(a.beta, c.x, v[0]);
      v[1] = fmaf(a.beta, c.y, v[1]);
      v[2] = fmaf(a.beta, c.z, v[2]);
      v[3] = fmaf(a.beta, c.w, v[3]);
    }
    if (EPI) {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = finish(a, v[j], n + j);
    }
    *reinterpret_cast<float4*>(cp) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (n + j < a.N) {
        float r = v[j];
        if (beta_nz) r = fmaf(a.beta, cp[j], r);
        cp[j] = EPI ? finish(a, r, n + j) : r;
      }
    }
  }
}

// alpha * acc (+ beta * C_old, bias, activation) for this thread's 8 rows x
// TN columns of the C tile at (tm0, tn0).  With beta != 0 the old C of four
// rows' quads is loaded before any of them is stored: as far as the compiler
// knows a store to C may alias a later load from C, so the load-store pairs
// of store_quad alone would wait out the memory latency once per quad (32
// times per wide tile, with one CTA per SM and nothing else to run).
template <int TN, bool EPI>
__device__ __forceinline__ void store_tile(const GemmArgs& a, int c_vec, long long tm0, long long tn0,
                                           int wm, int wn, int tm, int tn,
                                           const uint64_t (&acc)[8][TN / 2]) {
  constexpr int WN = SimtCfg<TN>::WN;
  constexpr int ROWS = TN == 16 ? 4 : 2;   // rows of quads loaded per batch (registers allowing)
  const bool beta_nz = a.beta != 0.f;
  const float* C = static_cast<const float*>(a.C);
#pragma unroll
  for (int i0 = 0; i0 < 8; i0 += ROWS) {
    float4 old[ROWS][TN / 4];
#pragma unroll
    for (int ii = 0; ii < ROWS; ++ii) {
      const long long m = tm0 + wm * 64 + (i0 + ii) * 8 + tm;
#pragma unroll
      for (int h = 0; h < TN / 4; ++h) {
        const long long n = tn0 + wn * WN + h * 16 + tn * 4;
        old[ii][h] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (beta_nz && m < a.M && c_vec && n + 3 < a.N)
          old[ii][h] = *reinterpret_cast<const float4*>(C + m * a.ldc + n);
      }
    }
#pragma unroll
    for (int ii = 0; ii < ROWS; ++ii) {
      const int i = i0 + ii;
      const long long m = tm0 + wm * 64 + i * 8 + tm;
      if (m >= a.M) continue;
#pragma unroll
      for (int h = 0; h < TN / 4; ++h) {
        const long long n = tn0 + wn * WN + h * 16 + tn * 4;
        const float2 lo = unpack2(acc[i][2 * h]), hi = unpack2(acc[i][2 * h + 1]);
        float v[4] = {a.alpha * lo.x, a.alpha * lo.y, a.alpha * hi.x, a.alpha * hi.y};
        if (c_vec && n + 3 < a.N) {
          if (beta_nz) {
            v[0] = fmaf(a.beta, old[ii][h].x, v[0]);
            v[1] = fmaf(a.beta, old[ii][h].y, v[1]);
            v[2] = fmaf(a.beta, old[ii][h].z, v[2]);
            v[3] = fmaf(a.beta, old[ii][h].w, v[3]);
          }
          if (EPI) {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = finish(a, v[j], n + j);
          }
          *reinterpret_cast<float4*>(static_cast<float*>(a.C) + m * a.ldc + n) =
              make_float4(v[0], v[1], v[2], v[3]);
        } else {
          store_quad<EPI>(a, c_vec, m, n, v);   // ragged or unaligned: element by element
        }
      }
    }
  }
}

// Stream-K: the end of this CTA's share of one tile (the K-slice u is one
// of its slices of that tile).  Every warp handles its own 64 x 4*TN block of
// the tile, so no barrier of the whole CTA is needed.  Returns false after a
// bounded wait ran out (the kernel's abort path follows).
template <int TN, bool EPI>
__device__ __forceinline__ bool sk_segment_end(const SimtParams& p, long long u, int k_slices, int tm0,
                                               int tn0, int warp, int lane,
                                               uint64_t (&acc)[8][TN / 2], volatile int* abort_flag) {
  using Cfg = SimtCfg<TN>;
  constexpr int BN = Cfg::BN, WN = Cfg::WN;
  const GemmArgs& a = p.a;
  const long long U = p.sk_units;
  const int G = p.sk_ctas;
  const long long T0 = u - u % k_slices, T1 = T0 + k_slices;   // this tile's K-slices
  int cfirst, clast, fin;
  sk_tile_workers(T0, T1, U, G, &cfirst, &clast, &fin);
  auto slot_of = [&](int c) {
    return c * kSkMaxSeg + (int)(T0 / k_slices - sk_begin(c, U, G) / k_slices);
  };
  const int me = (int)blockIdx.x;
  const int wm = warp / 4, wn = warp % 4, tm = lane % 8, tn = lane / 8;
  if (me != fin) {
    // ------------------------------------------------ contributor
    float* dst = p.sk_partials + (size_t)slot_of(me) * (BM * BN);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int h = 0; h < TN / 4; ++h) {
        const int row = wm * 64 + i * 8 + tm, col = wn * WN + h * 16 + tn * 4;
        const float2 lo = unpack2(acc[i][2 * h]), hi = unpack2(acc[i][2 * h + 1]);
        *reinterpret_cast<float4*>(dst + (size_t)row * BN + col) = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_u32(p.sk_flags + slot_of(me) * 8 + warp, 1u);
  } else {
    // ------------------------------------------------ finisher
    // every other part of this warp's block must be written (bounded wait)
    bool ok = true;
    if (lane == 0) {
      for (int c = cfirst; ok && c <= clast; ++c) {
        if (c == me) continue;
        const unsigned* flag = p.sk_flags + slot_of(c) * 8 + warp;
        if (ld_acquire_u32(flag) != 0u) continue;
        const uint64_t t0 = globaltimer_ns();
        while (true) {
          bool got = false;
#pragma unroll 1
          for (int r = 0; r < 32 && !got; ++r) got = ld_acquire_u32(flag) != 0u;
          if (got) break;
          if (*abort_flag || globaltimer_ns() - t0 > a.timeout_ns) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) {
        if (!*abort_flag) report_status(a.status, 5, kSiteSimtStreamK);
        *abort_flag = 1;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) return false;
    __syncwarp();
    __threadfence();
    // this CTA's part first, then the others in CTA order (fixed for the
    // shape, so every call gives the same bits); L2 loads (the parts were
    // written by other SMs)
    for (int c = cfirst; c <= clast; ++c) {
      if (c == me) continue;
      const float* src = p.sk_partials + (size_t)slot_of(c) * (BM * BN);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) {
          const int row = wm * 64 + i * 8 + tm, col = wn * WN + h * 16 + tn * 4;
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (size_t)row * BN + col));
          float2 lo = unpack2(acc[i][2 * h]), hi = unpack2(acc[i][2 * h + 1]);
          lo.x += v.x;
          lo.y += v.y;
          hi.x += v.z;
          hi.y += v.w;
          acc[i][2 * h] = pack2(lo.x, lo.y);
          acc[i][2 * h + 1] = pack2(hi.x, hi.y);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      for (int c = cfirst; c <= clast; ++c)
        if (c != me) p.sk_flags[slot_of(c) * 8 + warp] = 0u;   // ready for the next call
    }
    store_tile<TN, EPI>(a, p.c_vec, tm0, tn0, wm, wn, tm, tn, acc);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < TN / 2; ++q) acc[i][q] = 0ull;
  return true;
}

// TN: register-tile width (SimtCfg).
// EPI: bias and/or activation present (the plain instance has no trace of
// them, so the common case keeps the main loop's register allocation).
// SPLIT: CTAs of a cluster that share one C tile's K range (1: a whole tile
// per CTA); cluster rank r takes the r-th of SPLIT contiguous K ranges.
// SPLIT == 0 is the stream-K launch: the K-slices of the tiles from
// tile_base on, in tile order, are split evenly over the CTAs, so a tile's
// K range may be shared by CTAs of different clusters.  Each CTA leaves the
// partial sum of a tile it does not finish in the workspace and raises one
// flag per warp; the tile's finisher -- the CTA whose share of it ends
// latest within its own range -- adds the parts in CTA order (the same order
// whichever CTA finishes, so the result is deterministic), applies the
// epilogue and lowers the flags.  Only finishers wait, with a bound, on
// flags of CTAs that never wait; the grid never has more CTAs than fit at
// once.
// TRIGGER: a split launch of the last wave follows on the stream (the plain
// instance has no trace of it: its code runs at the original speed).
template <int TN, bool EPI, int SPLIT, bool TRIGGER>
__global__ void __launch_bounds__(THREADS, SimtCfg<TN>::CTAS_PER_SM)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap mapA,
                     const __grid_constant__ CUtensorMap mapB, const SimtParams p) {
  using Cfg = SimtCfg<TN>;
  constexpr int BN = Cfg::BN, WN = Cfg::WN, STAGES = Cfg::STAGES;
  constexpr int STAGE_BYTES = Cfg::STAGE_BYTES, A_STAGE_BYTES = Cfg::A_STAGE_BYTES;
  constexpr int PART_LD = Cfg::PART_LD;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t bar_base = base + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + STAGES * STAGE_BYTES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + STAGES);
  // per slot: warps done with it this round, and copies issued into it so far
  uint32_t* done_cnt = reinterpret_cast<uint32_t*>(bars + STAGES) + 4;
  uint32_t* issue_cnt = done_cnt + STAGES;
  const uint32_t stall_bar = bar_base + 192u;  // test hook: nothing arrives
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto a_tile = [&](int s) { return base + s * STAGE_BYTES; };
  auto b_tile = [&](int s) { return base + s * STAGE_BYTES + A_STAGE_BYTES; };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const GemmArgs& a = p.a;
  constexpr bool SK = SPLIT == 0;

  // Grouped raster over C tiles: groups of 16 row-panels, column-panel by
  // column-panel, so the CTAs in flight at one time cover a near-square
  // block of C and the A and B panels they share stay in L2 (4096^3 with
  // 128 x 128 tiles: 16 x 19 tiles, 32 MB of A and 38 MB of B; groups of 8
  // rows kept all of B in flight and read 19 % more from DRAM).
  auto tile_origin = [&](int tile, int& tm0, int& tn0) {
    const int group = 16;
    const int tiles_in_group = group * p.tiles_n;
    const int g = tile / tiles_in_group;
    const int first_m = g * group;
    const int gsize = min(p.tiles_m - first_m, group);
    tm0 = (first_m + (tile % tiles_in_group) % gsize) * BM;
    tn0 = ((tile % tiles_in_group) / gsize) * BN;
  };
  const int k_slices = (a.K + BK - 1) / BK;   // K-slices of one tile
  int m0, n0, k_tiles = k_slices, kt_first = 0, part = 0;
  // stream-K: this CTA's range starts at K-slice k_first of tile sk_tile and
  // is at most one tile long, so it ends in that tile or the next one
  // (origin m1, n1); seg_end is the last range index inside the first tile
  long long u0 = 0;
  int sk_tile = 0, seg_end = 0, m1 = 0, n1 = 0;
  if constexpr (SK) {
    u0 = sk_begin(blockIdx.x, p.sk_units, p.sk_ctas);
    k_tiles = (int)(sk_begin(blockIdx.x + 1, p.sk_units, p.sk_ctas) - u0);
    sk_tile = (int)(u0 / k_slices);
    kt_first = (int)(u0 - (long long)sk_tile * k_slices);
    seg_end = k_slices - kt_first - 1;
    tile_origin(p.tile_base + sk_tile, m0, n0);
    if (seg_end < k_tiles - 1) tile_origin(p.tile_base + sk_tile + 1, m1, n1);
  } else {
    tile_origin(SPLIT > 1 ? p.tile_base + (int)(blockIdx.x / SPLIT) : (int)blockIdx.x, m0, n0);
  }
  if constexpr (SPLIT > 1) {
    part = (int)cluster_ctarank();
    kt_first = k_tiles * part / SPLIT;
    k_tiles = k_tiles * (part + 1) / SPLIT - kt_first;
  }
  // The i-th K-slice this CTA streams: its A and B coordinates.
  auto slice_coords = [&](int i, int& xk, int& ym, int& xn) {
    if constexpr (SK) {
      const bool second = i > seg_end;
      ym = second ? m1 : m0;
      xn = second ? n1 : n0;
      xk = (second ? i - seg_end - 1 : kt_first + i) * BK;
    } else {
      ym = m0;
      xn = n0;
      xk = (kt_first + i) * BK;
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      done_cnt[s] = 0;
      issue_cnt[s] = 0;
    }
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // the split launch of the last wave may take SM slots as this grid's CTAs
    // leave (it reads nothing this grid writes)
    if constexpr (TRIGGER) griddep_launch_dependents();
  }
  __syncthreads();

  // Thread 0 issues the first STAGES K-slices; every later copy is issued by
  // the last warp to release its slot.  (A dedicated producer warp would put
  // five warps on one scheduler at two CTAs per SM and cap registers at 96.)
  const bool producer = threadIdx.x == 0;
  if (producer) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
    for (int kt = 0; kt < k_tiles && kt < STAGES; ++kt) {
      int xk, ym, xn;
      slice_coords(kt, xk, ym, xn);
      mbar_arrive_expect_tx(full_bar(kt), STAGE_BYTES);
      tma_load_2d(a_tile(kt), &mapA, full_bar(kt), xk, ym);
      tma_load_2d(b_tile(kt), &mapB, full_bar(kt), xn, xk);
      issue_cnt[kt] = 1;
    }
  }

  // Warp (wm, wn) owns rows 64*wm .. +64 and columns WN*wn .. +WN of the C
  // tile; lane (tm, tn) owns rows 64*wm + 8*i + tm (i < 8) and the columns
  // WN*wn + 16*h + 4*tn .. +4 (h < TN/4).
  const int wm = warp / 4, wn = warp % 4;
  const int tm = lane % 8, tn = lane / 8;
  const int sw = (tm >> 1) & 3;                // 64-byte swizzle phase of my rows
  const uint32_t a_row_off = (uint32_t)(wm * 64 + tm) * 64u;
  const uint32_t b_col_off = (uint32_t)(wn * WN + tn * 4) * 4u;
  // acc[i][q] holds C columns (2q, 2q+1) of my TN columns, row i
  uint64_t acc[8][TN / 2];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < TN / 2; ++q) acc[i][q] = 0ull;

  bool ok = true;
  int my_k_tiles = k_tiles;
  if (a.stall && warp == 0 && blockIdx.x == 0 && k_tiles > 0) {
    // test hook: warp 0 of the first CTA waits on a barrier nothing arrives
    // at, so its bounded wait runs out and the abort path runs
    if (!mbar_wait(stall_bar, 0, a.timeout_ns / 4, abort_flag)) {
      if (!*abort_flag) report_status(a.status, 5, kSiteSimtConsumer);
      *abort_flag = 1;
      ok = false;
      my_k_tiles = 0;
    }
  }
  // The K-slices run in pieces: one for a whole tile or a split part; for
  // stream-K, the slices of the range inside its first tile, then those in
  // the next tile, each piece followed by its hand-over or finish, so the
  // per-slice loop carries no test for a piece's end.
#pragma unroll 1
  for (int piece = 0; piece < (SK ? 2 : 1); ++piece) {
    const int kt_lo = piece == 0 ? 0 : seg_end + 1;
    const int kt_hi = SK && piece == 0 ? min(seg_end + 1, my_k_tiles) : my_k_tiles;
    for (int kt = kt_lo; kt < kt_hi; ++kt) {
      const int s = kt % STAGES;
      const uint32_t parity = (uint32_t)(kt / STAGES) & 1u;
      if (!mbar_wait(full_bar(s), parity, a.timeout_ns, abort_flag)) {
        if (!*abort_flag) report_status(a.status, 5, kSiteSimtConsumer);
        *abort_flag = 1;
        ok = false;
        break;
      }
      const uint32_t at = a_tile(s) + a_row_off;
      const uint32_t bt = b_tile(s) + b_col_off;
#pragma unroll
      for (int kp = 0; kp < BK / 2; ++kp) {
        // rows i*8+tm, k = 2kp, 2kp+1: one 8-byte load per row inside the
        // swizzled 16-byte chunk that holds k = 4*(kp/2) .. 4*(kp/2)+3
        // (loading the next pair's values a step ahead was 2 % slower)
        const uint32_t off = (uint32_t)((((kp >> 1) ^ sw) * 16) + (kp & 1) * 8);
        float2 av[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) av[i] = lds64(at + i * 8 * 64 + off);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint32_t brow = bt + (uint32_t)(kp * 2 + kk) * (BN * 4);
          uint64_t b[TN / 2];
#pragma unroll
          for (int h = 0; h < TN / 4; ++h) lds_pairs(brow + h * 64, b[2 * h], b[2 * h + 1]);
          if constexpr (TN == 8 && EPI) {
            // rows outer: the 8 x 8 instance with an epilogue would spill at
            // 128 registers with all eight broadcasts live at once
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint64_t a2 = dup2(kk == 0 ? av[i].x : av[i].y);
#pragma unroll
              for (int q = 0; q < TN / 2; ++q) ffma2(acc[i][q], a2, b[q]);
            }
          } else {
            uint64_t a2[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a2[i] = dup2(kk == 0 ? av[i].x : av[i].y);
            // B pair outer, rows inner: consecutive FMAs share the B operand
#pragma unroll
            for (int q = 0; q < TN / 2; ++q)
#pragma unroll
              for (int i = 0; i < 8; ++i) ffma2(acc[i][q], a2[i], b[q]);
          }
        }
      }
      __syncwarp();  // every lane of this warp is done reading slot s
      if (lane == 0) {
        // the last of the eight warps to release slot s refills it with K-slice
        // kt+STAGES; the slot's next round cannot start before that copy lands
        __threadfence_block();
        if (atomicAdd(&done_cnt[s], 1u) == COMPUTE_WARPS - 1) {
          done_cnt[s] = 0;
          __threadfence_block();
          if (kt + STAGES < k_tiles && !*abort_flag) {
            int xk, ym, xn;
            slice_coords(kt + STAGES, xk, ym, xn);
            mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
            tma_load_2d(a_tile(s), &mapA, full_bar(s), xk, ym);
            tma_load_2d(b_tile(s), &mapB, full_bar(s), xn, xk);
            atomicAdd(&issue_cnt[s], 1u);
          }
        }
      }
    }
    if (!ok) break;
    if constexpr (SK) {
      // ------------------------------------------ stream-K piece end
      if (kt_hi > kt_lo &&
          !sk_segment_end<TN, EPI>(p, u0 + kt_lo, k_slices, piece ? m1 : m0, piece ? n1 : n0, warp,
                                   lane, acc, abort_flag)) {
        ok = false;
        break;
      }
    }
  }
  __syncthreads();  // every warp has left the main loop
  if (producer && *abort_flag) {
    // every copy already issued must land before shared memory is released:
    // the latest copy into slot s completes its phase issue_cnt[s] - 1
    for (int s = 0; s < STAGES; ++s)
      if (issue_cnt[s] > 0 &&
          !mbar_wait(full_bar(s), (issue_cnt[s] - 1u) & 1u, kDrainWaitNs, nullptr))
        report_status(a.status, 5, kSiteSimtDrain);
  }

  if constexpr (SPLIT == 1) {
    if (ok) store_tile<TN, EPI>(a, p.c_vec, m0, n0, wm, wn, tm, tn, acc);   // epilogue
  } else if constexpr (SPLIT > 1) {
    // ------------------------------------------- split epilogue (cluster)
    // Every copy this CTA issued has landed (all were consumed, or drained
    // above), so the ring holds this CTA's partial tile.
    if (!*abort_flag) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) {
          const int row = wm * 64 + i * 8 + tm, col = wn * WN + h * 16 + tn * 4;
          const float2 lo = unpack2(acc[i][2 * h]), hi = unpack2(acc[i][2 * h + 1]);
          *reinterpret_cast<float4*>(base_ptr + ((size_t)row * PART_LD + col) * 4) =
              make_float4(lo.x, lo.y, hi.x, hi.y);
        }
      }
    }
    cluster_sync();  // every rank's partial (and abort flag) is written
    bool all_ok = true;
#pragma unroll
    for (int r = 0; r < SPLIT; ++r)
      all_ok &= ld_dsmem_u32(map_to_rank(bar_base + 8u * STAGES, (uint32_t)r)) == 0u;
    if (all_ok) {
      // rank `part` sums rows [part*BM/SPLIT, (part+1)*BM/SPLIT) over the
      // ranks in order 0..SPLIT-1, in chunks of QC quads per thread (all
      // of a chunk's loads in flight before the first add)
      constexpr int QUADS = (BM / SPLIT) * (BN / 4) / THREADS;
      constexpr int QC = QUADS < 4 ? QUADS : 4;
      static_assert(QUADS % QC == 0 && (BM / SPLIT) * (BN / 4) % THREADS == 0, "reduce split");
#pragma unroll 1
      for (int q0 = 0; q0 < QUADS; q0 += QC) {
        float4 t[QC][SPLIT];
#pragma unroll
        for (int q = 0; q < QC; ++q) {
          const int idx = (int)threadIdx.x + (q0 + q) * THREADS;
          const int row = part * (BM / SPLIT) + idx / (BN / 4), col = (idx % (BN / 4)) * 4;
          const uint32_t off = base + (uint32_t)(row * PART_LD + col) * 4u;
#pragma unroll
          for (int r = 0; r < SPLIT; ++r) t[q][r] = ld_dsmem_f32x4(map_to_rank(off, (uint32_t)r));
        }
#pragma unroll
        for (int q = 0; q < QC; ++q) {
          const int idx = (int)threadIdx.x + (q0 + q) * THREADS;
          const long long m = (long long)m0 + part * (BM / SPLIT) + idx / (BN / 4);
          const long long n = (long long)n0 + (idx % (BN / 4)) * 4;
          float4 sum = t[q][0];
#pragma unroll
          for (int r = 1; r < SPLIT; ++r) {
            sum.x += t[q][r].x;
            sum.y += t[q][r].y;
            sum.z += t[q][r].z;
            sum.w += t[q][r].w;
          }
          float v[4] = {a.alpha * sum.x, a.alpha * sum.y, a.alpha * sum.z, a.alpha * sum.w};
          if (m < a.M) store_quad<EPI>(a, p.c_vec, m, n, v);
        }
      }
    }
    cluster_sync();  // no rank leaves while another still reads its partial
    // A grid that finishes before the one it overlaps would let later work on
    // the stream run early; completion waits for that grid.
    griddep_wait();
  } else {
    // stream-K: every segment was finished or handed over inside the loop;
    // as for the cluster split, completion waits for the grid it overlaps
    griddep_wait();
  }
  __syncthreads();
}

// Resident clusters of four CTAs of the narrow configuration's split kernel,
// per device (a GPC whose free CTA slots are not a multiple of four leaves
// the rest idle); queried once, the EPI instances having the same resources.
struct SimtDeviceInfo {
  std::atomic<bool> ready{false};   // published after the field below is set
  int max_clusters4 = 0;
};

cudaError_t narrow_clusters4(int num_sms, int* c4) {
  using Cfg = SimtCfg<8>;
  static SimtDeviceInfo info[64];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!info[dev].ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!info[dev].ready.load(std::memory_order_relaxed)) {
      auto k = sgemm_tma_kernel<8, false, 4, false>;
      if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES)) !=
          cudaSuccess)
        return e;
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 4;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.blockDim = dim3(THREADS, 1, 1);
      cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      cfg.gridDim = dim3((unsigned)(4 * Cfg::CTAS_PER_SM * num_sms), 1, 1);
      int n = 0;
      if ((e = cudaOccupancyMaxActiveClusters(&n, k, &cfg)) != cudaSuccess) return e;
      info[dev].max_clusters4 = n;
      info[dev].ready.store(true, std::memory_order_release);
    }
  }
  *c4 = info[dev].max_clusters4;
  return cudaSuccess;
}

// The stream-K workspace of a device, shared with the CTA-pair tensor-core
// kernel: kSkSlots slots, each with room for the partial tiles and flags of
// a stream-K launch of up to one CTA per SM (152 SMs: 39.8 MB of partials a
// slot; the same room holds two 256 x 256 partial tiles per SM pair),
// allocated and zeroed at the first call of either kernel on the device and
// kept until the process exits.  Calls take the slots in turn, so up to
// kSkSlots stream-K calls may run on the GPU at once (on different streams)
// without sharing one.
constexpr int kSkSlots = 4;
struct SkWorkspace {
  std::atomic<bool> ready{false};   // published after the fields below are set
  float* partials = nullptr;        // kSkSlots x slot_floats
  unsigned* flags = nullptr;        // kSkSlots x slot_flags, zero between calls
  size_t slot_floats = 0, slot_flags = 0;
  int max_ctas = 0;
  std::atomic<unsigned> next{0};
};
SkWorkspace g_sk[64];
std::mutex g_sk_mu;

cudaError_t sk_workspace(int num_sms, SkWorkspace** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SkWorkspace& w = g_sk[dev];
  if (!w.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_sk_mu);
    if (!w.ready.load(std::memory_order_relaxed)) {
      using Cfg = SimtCfg<16>;
      const int ctas = Cfg::CTAS_PER_SM * num_sms;
      const size_t slot_floats = (size_t)ctas * kSkMaxSeg * BM * Cfg::BN;
      const size_t slot_flags = (size_t)ctas * kSkMaxSeg * COMPUTE_WARPS;
      void* p = nullptr;
      if ((e = cudaMalloc(&p, kSkSlots * slot_floats * sizeof(float))) != cudaSuccess) return e;
      void* f = nullptr;
      if ((e = cudaMalloc(&f, kSkSlots * slot_flags * sizeof(unsigned))) != cudaSuccess) {
        cudaFree(p);
        return e;
      }
      if ((e = cudaMemset(f, 0, kSkSlots * slot_flags * sizeof(unsigned))) != cudaSuccess ||
          (e = cudaDeviceSynchronize()) != cudaSuccess) {
        cudaFree(p);
        cudaFree(f);
        return e;
      }
      w.partials = static_cast<float*>(p);
      w.flags = static_cast<unsigned*>(f);
      w.slot_floats = slot_floats;
      w.slot_flags = slot_flags;
      w.max_ctas = ctas;
      w.ready.store(true, std::memory_order_release);
    }
  }
  *out = &w;
  return cudaSuccess;
}

}  // namespace

cudaError_t stream_k_setup(int num_sms) {
  SkWorkspace* w = nullptr;
  return sk_workspace(num_sms, &w);
}

cudaError_t stream_k_slot(int num_sms, float** partials, unsigned** flags, size_t* slot_floats,
                          size_t* slot_flags) {
  SkWorkspace* w = nullptr;
  const cudaError_t e = sk_workspace(num_sms, &w);
  if (e != cudaSuccess) return e;
  const unsigned slot = w->next.fetch_add(1, std::memory_order_relaxed) % kSkSlots;
  *partials = w->partials + slot * w->slot_floats;
  *flags = w->flags + slot * w->slot_flags;
  *slot_floats = w->slot_floats;
  *slot_flags = w->slot_flags;
  return cudaSuccess;
}

namespace {

// CTAs of a stream-K launch for `rest` tiles of k_slices K-slices each: one
// per SM at most, each with at least kSkMinSlices K-slices (two rounds of the
// ring), so a CTA's range is at most one tile long when k_slices >= kSkMinSlices.
constexpr int kSkMinSlices = 2 * SimtCfg<16>::STAGES;
int sk_ctas(long long rest, int k_slices, int num_sms) {
  const long long by_work = rest * k_slices / kSkMinSlices;
  const long long g = by_work < num_sms ? by_work : num_sms;
  return (int)(g < 1 ? 1 : g);
}

// The stream-K launch and the largest number of CTAs that share one tile.
template <bool EPI>
cudaError_t launch_stream_k(const CUtensorMap* mapA, const CUtensorMap* mapB, SimtParams p,
                            long long rest, int k_slices, int num_sms, bool overlap, cudaStream_t s,
                            int* max_share) {
  using Cfg = SimtCfg<16>;
  static std::atomic<uint64_t> smem_set{0};
  auto k = sgemm_tma_kernel<16, EPI, 0, false>;
  cudaError_t e = set_smem_once(smem_set, k, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int G = sk_ctas(rest, k_slices, num_sms);
  float* partials = nullptr;
  unsigned* flags = nullptr;
  size_t slot_floats = 0, slot_flags = 0;
  if ((e = stream_k_slot(num_sms, &partials, &flags, &slot_floats, &slot_flags)) != cudaSuccess) return e;
  if ((size_t)G * kSkMaxSeg * BM * Cfg::BN > slot_floats || (size_t)G * kSkMaxSeg * COMPUTE_WARPS > slot_flags)
    return cudaErrorInvalidValue;
  p.sk_units = rest * k_slices;
  p.sk_ctas = G;
  p.sk_partials = partials;
  p.sk_flags = flags;
  *max_share = sk_max_share(rest, k_slices, G);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)G, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  // overlap the first launch's last CTAs only when there is one: otherwise
  // the previous kernel on the stream may still be writing A, B or C
  cfg.numAttrs = overlap ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, k, *mapA, *mapB, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The split launch: `units` C tiles (the tiles past the last whole wave),
// each K-split over a cluster of SPLIT CTAs.  overlap: a first launch
// precedes it on the stream and triggers it early.
template <int TN, bool EPI, int SPLIT>
cudaError_t launch_split(const CUtensorMap* mapA, const CUtensorMap* mapB, const SimtParams& p,
                         long long units, bool overlap, cudaStream_t s) {
  using Cfg = SimtCfg<TN>;
  static std::atomic<uint64_t> smem_set{0};
  auto k = sgemm_tma_kernel<TN, EPI, SPLIT, false>;
  cudaError_t e = set_smem_once(smem_set, k, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)SPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  attr[1].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
  attr[2].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[2].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.gridDim = dim3((unsigned)(units * SPLIT), 1, 1);
  // The hardware may place a cluster's CTAs where slots are free (4096^3 on
  // GB300 with 128 x 128 tiles: 2.352 -> 2.272 ms against the default
  // placement).  Overlap the first launch's last CTAs only when there is
  // one: otherwise the previous kernel on the stream may still be writing A,
  // B or C.
  cfg.numAttrs = overlap ? 3 : 2;
  e = cudaLaunchKernelEx(&cfg, k, *mapA, *mapB, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int TN, bool EPI>
cudaError_t launch_plan(const CUtensorMap* mapA, const CUtensorMap* mapB, SimtParams p,
                        long long tiles, const SimtPlan& plan, int num_sms, cudaStream_t s,
                        int* k_split) {
  using Cfg = SimtCfg<TN>;
  static std::atomic<uint64_t> smem_whole{0}, smem_first{0};
  auto whole_kernel = sgemm_tma_kernel<TN, EPI, 1, false>;
  auto first_kernel = sgemm_tma_kernel<TN, EPI, 1, true>;
  cudaError_t e = set_smem_once(smem_whole, whole_kernel, Cfg::SMEM_BYTES);
  if (e == cudaSuccess) e = set_smem_once(smem_first, first_kernel, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  *k_split = 1;
  if (plan.split == 1) {
    whole_kernel<<<(unsigned)tiles, THREADS, Cfg::SMEM_BYTES, s>>>(*mapA, *mapB, p);
    return cudaGetLastError();
  }
  const long long slots = (long long)Cfg::CTAS_PER_SM * num_sms;
  const long long rest = tiles % slots, whole = tiles - rest;
  if (rest == 0) return cudaErrorInvalidValue;  // the plan splits only a partial wave
  if (whole > 0) {
    first_kernel<<<(unsigned)whole, THREADS, Cfg::SMEM_BYTES, s>>>(*mapA, *mapB, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  p.tile_base = (int)whole;
  if constexpr (TN == 16) {  // the wide tile's tail runs stream-K
    if (plan.split != 0) return cudaErrorInvalidValue;
    const int k_slices = (p.a.K + BK - 1) / BK;
    return launch_stream_k<EPI>(mapA, mapB, p, rest, k_slices, num_sms, whole > 0, s, k_split);
  } else {
    if (plan.split != 4) return cudaErrorInvalidValue;
    *k_split = 4;
    return launch_split<TN, EPI, 4>(mapA, mapB, p, rest, whole > 0, s);
  }
}

// The wave model's estimate for one configuration (plan::simt_option), after
// the occupancy query it needs.
template <int TN>
cudaError_t option_for(long long tiles, int k_tiles, int num_sms, bool split_allowed,
                       plan::SimtOption* o) {
  using Cfg = SimtCfg<TN>;
  int c4 = 0;
  const long long slots = (long long)Cfg::CTAS_PER_SM * num_sms;
  const int min_k_tiles = 2 * Cfg::STAGES;  // two rounds of the ring per rank
  // a cheap first test before the occupancy query (the wide tile's stream-K
  // tail needs none)
  if (TN == 8 && split_allowed && tiles % slots != 0 && k_tiles >= 4 * min_k_tiles) {
    const cudaError_t e = narrow_clusters4(num_sms, &c4);
    if (e != cudaSuccess) return e;
  }
  *o = plan::simt_option(TN, tiles, k_tiles, num_sms, 0, c4, min_k_tiles, split_allowed);
  return cudaSuccess;
}

}  // namespace

int plan_f32_simt(int M, int N, int K, int num_sms, int forced_tn, SimtPlan* out) {
  const long long tiles_m = (M + BM - 1) / BM;
  const long long tiles8 = tiles_m * ((N + kSimtBN8 - 1) / kSimtBN8);
  const long long tiles16 = tiles_m * ((N + kSimtBN16 - 1) / kSimtBN16);
  const int k_tiles = (K + BK - 1) / BK;
  const bool allowed = split_tiles_enabled();
  plan::SimtOption o8{}, o16{};
  cudaError_t e;
  if (forced_tn != 16 && (e = option_for<8>(tiles8, k_tiles, num_sms, allowed, &o8)) != cudaSuccess) return e;
  if (forced_tn != 8 && (e = option_for<16>(tiles16, k_tiles, num_sms, allowed, &o16)) != cudaSuccess)
    return e;
  // the wide tiles must win by the model's margin of error (2560 x 2048 x
  // 1024 on GB300: estimated 4 % faster wide, measured 7 % slower)
  const bool wide = forced_tn == 16 || (forced_tn != 8 && o16.time < plan::kSimtWideMargin * o8.time);
  out->tn = wide ? 16 : 8;
  out->split = wide ? o16.split : o8.split;
  return cudaSuccess;
}

int launch_f32_simt(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                    const SimtPlan& plan, int num_sms, cudaStream_t s, int* k_split) {
  *k_split = 1;
  SimtParams p;
  p.a = a;
  const int bn = plan.tn == 16 ? kSimtBN16 : kSimtBN8;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = (a.N + bn - 1) / bn;
  p.c_vec = ((reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && (a.ldc % 4) == 0) ? 1 : 0;
  p.tile_base = 0;
  const long long tiles = (long long)p.tiles_m * p.tiles_n;
  if (tiles <= 0) return cudaSuccess;
  if (tiles * 4 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.sk_units = 0;
  p.sk_ctas = 0;
  p.sk_partials = nullptr;
  p.sk_flags = nullptr;
  const bool epi = a.bias != nullptr || a.act != kActNone;
  if (plan.tn == 16)
    return epi ? launch_plan<16, true>(mapA, mapB, p, tiles, plan, num_sms, s, k_split)
               : launch_plan<16, false>(mapA, mapB, p, tiles, plan, num_sms, s, k_split);
  if (plan.tn == 8)
    return epi ? launch_plan<8, true>(mapA, mapB, p, tiles, plan, num_sms, s, k_split)
               : launch_plan<8, false>(mapA, mapB, p, tiles, plan, num_sms, s, k_split);
  return cudaErrorInvalidValue;
}

void sk_clear_flags() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
  SkWorkspace& w = g_sk[dev];
  if (w.ready.load(std::memory_order_acquire))
    cudaMemset(w.flags, 0, kSkSlots * w.slot_flags * sizeof(unsigned));
}

// ------------------------------------------------------ gemm_f32_noalloc
// The scratch of gemm_f32_noalloc: the partial tiles (kSkMaxSeg per CTA,
// 128 x 256 floats each) and the per-warp release flags of one stream-K tail
// of up to kStaticScratchCtas CTAs -- 38 MiB of partials and 9.5 KB of
// flags, reserved on each device when this file's module loads rather than
// allocated by a call.  There is one per device: two calls that execute on
// one device at the same time share it and race.
constexpr size_t kStaticPartialFloats = (size_t)kStaticScratchCtas * kSkMaxSeg * BM * kSimtBN16;
constexpr size_t kStaticFlagWords = (size_t)kStaticScratchCtas * kSkMaxSeg * COMPUTE_WARPS;
static_assert(kStaticPartialFloats % 64 == 0, "flags start on a 256-byte boundary");
static __device__ __align__(256) float g_static_scratch[kStaticPartialFloats + kStaticFlagWords];

namespace {

struct StaticScratch {
  std::atomic<bool> ready{false};   // published after `base` is set
  float* base = nullptr;
};
StaticScratch g_static[64];
std::mutex g_static_mu;

// Set-up, once per device with that device current: the array's device
// address (no allocation; nothing is launched).
cudaError_t static_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  StaticScratch& st = g_static[dev];
  if (!st.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!st.ready.load(std::memory_order_relaxed)) {
      float* ptr = nullptr;
      e = cudaGetSymbolAddress((void**)&ptr, g_static_scratch);
      if (e != cudaSuccess) return e;
      if (ptr == nullptr) return cudaErrorInvalidSymbol;
      st.base = ptr;
      st.ready.store(true, std::memory_order_release);
    }
  }
  *out = st.base;
  return cudaSuccess;
}

}  // namespace

size_t simt_static_scratch_bytes() { return sizeof(float) * (kStaticPartialFloats + kStaticFlagWords); }

int simt_stream_k_ctas(int M, int N, int K, const SimtPlan& plan, int num_sms) {
  if (plan.tn != 16 || plan.split != 0 || M <= 0 || N <= 0 || num_sms <= 0) return 0;
  const long long tiles = (long long)((M + BM - 1) / BM) * ((N + kSimtBN16 - 1) / kSimtBN16);
  const long long rest = tiles % ((long long)SimtCfg<16>::CTAS_PER_SM * num_sms);
  if (rest == 0) return 0;
  return sk_ctas(rest, (K + BK - 1) / BK, num_sms);
}

int launch_f32_simt_static(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                           const SimtPlan& plan, int num_sms, cudaStream_t s, int* k_split) {
  *k_split = 1;
  if (a.bias != nullptr || a.act != kActNone) return cudaErrorInvalidValue;
  float* scratch = nullptr;
  cudaError_t e = static_scratch(&scratch);
  if (e != cudaSuccess) return e;
  SimtParams p;
  p.a = a;
  const int bn = plan.tn == 16 ? kSimtBN16 : kSimtBN8;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = (a.N + bn - 1) / bn;
  p.c_vec = ((reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && (a.ldc % 4) == 0) ? 1 : 0;
  p.tile_base = 0;
  p.sk_units = 0;
  p.sk_ctas = 0;
  p.sk_partials = nullptr;
  p.sk_flags = nullptr;
  const long long tiles = (long long)p.tiles_m * p.tiles_n;
  if (tiles <= 0) return cudaSuccess;
  if (tiles * 4 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // the narrow tiles (whole waves, or clusters sharing a tile through
  // distributed shared memory) and wide tiles without a tail use no scratch
  if (plan.tn == 8) return launch_plan<8, false>(mapA, mapB, p, tiles, plan, num_sms, s, k_split);
  if (plan.tn != 16) return cudaErrorInvalidValue;
  if (plan.split == 1) return launch_plan<16, false>(mapA, mapB, p, tiles, plan, num_sms, s, k_split);
  if (plan.split != 0) return cudaErrorInvalidValue;

  // wide tiles: whole waves, then the stream-K tail on the static scratch
  using Cfg = SimtCfg<16>;
  static std::atomic<uint64_t> smem_first{0}, smem_sk{0};
  auto first_kernel = sgemm_tma_kernel<16, false, 1, true>;
  auto sk_kernel = sgemm_tma_kernel<16, false, 0, false>;
  if ((e = set_smem_once(smem_first, first_kernel, Cfg::SMEM_BYTES)) != cudaSuccess) return e;
  if ((e = set_smem_once(smem_sk, sk_kernel, Cfg::SMEM_BYTES)) != cudaSuccess) return e;
  const long long slots = (long long)Cfg::CTAS_PER_SM * num_sms;
  const long long rest = tiles % slots, whole = tiles - rest;
  if (rest == 0) return cudaErrorInvalidValue;  // the plan splits only a partial wave
  const int k_slices = (a.K + BK - 1) / BK;
  const int G = sk_ctas(rest, k_slices, num_sms);
  if (G > kStaticScratchCtas) return cudaErrorInvalidValue;
  unsigned* flags = reinterpret_cast<unsigned*>(scratch + kStaticPartialFloats);
  // the flags must be zero when the tail starts: cleared on this stream
  // before the first launch, so a call after one that timed out (and left
  // flags raised) starts clean
  e = cudaMemsetAsync(flags, 0, (size_t)G * kSkMaxSeg * COMPUTE_WARPS * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  if (whole > 0) {
    first_kernel<<<(unsigned)whole, THREADS, Cfg::SMEM_BYTES, s>>>(*mapA, *mapB, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  p.tile_base = (int)whole;
  p.sk_units = rest * k_slices;
  p.sk_ctas = G;
  p.sk_partials = scratch;
  p.sk_flags = flags;
  *k_split = sk_max_share(rest, k_slices, G);   // the most CTAs that meet in one tile
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)G, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = whole > 0 ? 1 : 0;   // overlap the whole waves' end only after them
  e = cudaLaunchKernelEx(&cfg, sk_kernel, *mapA, *mapB, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace g3
