// BF16 GEMM on a CTA pair: the same computation as gemm_bf16_tc.cu with C
// tiles of 256 x BN computed by two CTAs (a cluster of two) that issue one
// M = 256 tcgen05.mma together (cta_group::2).
//
// Why: a single CTA computing 128 x 256 moves 48 KB per 64-deep K-stage into
// shared memory and the MMAs read all of it back.  In the pair each CTA loads
// its 128 rows of A and only half of B's columns, and the MMA reads A from
// each CTA and B from both, so every shared-memory and L2 byte feeds twice
// the FLOPs -- the per-stage A/B intensity of "Kernel 性能从何而来" (section
// "优化 Memory-Bound Kernel", blocking) rises from 2*128*256/(2*(128+256)) = 85
// to 2*256*256/(2*2*(128+128)) = 128 FLOP/byte per CTA.  Section "优化阶梯"
// of the same page names CTA clusters as the step after warp specialisation.
//
// Roles (192 threads per CTA, both CTAs): warp 0 = TMA producer (each CTA
// loads its own A rows and B columns; the copies of both CTAs complete on the
// leader CTA's barrier), warp 1 = TMEM allocation for the pair and, in the
// leader only, the single MMA-issuing thread, warps 2-5 = epilogue of the
// CTA's 128 rows.  The leader's commits arrive on both CTAs' barriers
// (multicast), and both CTAs' epilogues arrive on the leader's
// accumulator-empty barrier.  Waits are bounded as in the single-CTA kernel.
//
// Persistent schedule: tiles [0, dp_tiles) go to the pairs in turn.  When the
// last wave would be partial (R = tiles mod pairs) and 2R pairs exist, those R
// tiles instead run as 2R half-width items (256 x BN/2) on 2R pairs: a
// half-width tile costs about 0.58 of a full one (measured per-column costs
// of the 128- and 256-wide pair tiles), so the last wave shrinks from a whole
// tile-time to a bit over half of one, with nothing to reduce afterwards.
//
// SwiGLU variant (SW, BN = 256): C = silu(A*Bgate) * (A*Bup) on C tiles of
// 256 x 128.  Each CTA's half of the MMA's B operand is 64 columns of Bgate
// (box 0) and the same 64 columns of Bup (box 1), so the MMA is the 256-wide
// one above and accumulator column x holds output column
// n0 + 64*(x / 128) + x % 64 of the gate (x % 128 < 64) or of the up
// projection; the epilogue pairs them and applies silu(g) * u.  The
// intermediate products never leave the chip and A is read once for both.
//
// FP8 variant (F8, BN = 256): A and B hold 8-bit floats (E4M3 or E5M2 each,
// "Kernel 性能从何而来", section "优化 Memory-Bound Kernel": a narrower type
// moves fewer bytes per FLOP).  A K-stage is still one 128-byte swizzle row
// per operand row, now 128 elements deep, so stage sizes, the pipeline and
// the epilogue are the bf16 ones; each CTA loads one 128-column box of B, the
// MMA is kind::f8f6f4 with K = 32 per instruction, and there is no
// half-width tail (a half tile would need 64-column boxes).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "plan.h"
#include "ptx.cuh"
#include "stream_k.cuh"
#include "tc_epilogue.cuh"

namespace g3 {
namespace {

constexpr int BM_CTA = kTcBM;    // rows per CTA
constexpr int BM = 2 * BM_CTA;   // rows per pair tile
constexpr int TMEM_COLS = 512;
constexpr int NUM_EPI_WARPS = 4;
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_LIMIT = 232448;
// Tiles are rastered in groups of 16 row panels, column panel by column
// panel: the 76 pairs' tiles in flight then share A and B panels in L2
// (4096^3: 69 MB read from DRAM against 67 MB of A and B; groups of 8: 80 MB).
constexpr int RASTER_GROUP = 16;
constexpr uint64_t kDrainGraceNs = 50000;        // after an abort, time for the peer's copies to land
constexpr uint16_t kBothCtas = 0x3;

// Stage geometry: every operand row of a K-stage is one 128-byte swizzle row
// (64 bf16 or 128 FP8 elements of K); B boxes are 128 bytes wide in n.
template <bool F8>
struct Geom {
  static constexpr int ESIZE = F8 ? 1 : 2;
  static constexpr int BK = 128 / ESIZE;                 // K elements per stage
  static constexpr int UMMA_K = F8 ? 32 : 16;           // K per MMA instruction
  static constexpr int BOX_N = 128 / ESIZE;             // columns per B box
  static constexpr int A_STAGE_BYTES = BM_CTA * 128;    // 16 KB
  static constexpr int B_BOX_BYTES = BOX_N * BK * ESIZE;  // 8 KB bf16, 16 KB FP8
  static constexpr int A_KSTEP = UMMA_K * ESIZE;        // bytes per MMA along a K-major row
  static constexpr int B_KSTEP = UMMA_K * 128;          // bytes per MMA down N-major rows
};
static_assert(Geom<false>::BK == kTcBK && Geom<true>::BK == kF8BK, "K per stage");

template <int BN, bool F8 = false>
struct PairCfg {
  using G = Geom<F8>;
  static_assert(BN == 128 || BN == 256, "pair tiles are 128 or 256 wide");
  static_assert(!F8 || BN == 256, "FP8 tiles load one whole 128-column box per CTA");
  static constexpr int B_BOXES = BN / 2 / G::BOX_N;
  static constexpr int STAGE_BYTES = G::A_STAGE_BYTES + B_BOXES * G::B_BOX_BYTES;  // per CTA
  static constexpr int STAGES_FIT = (SMEM_LIMIT - BAR_BYTES - 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
};

template <int BN>
__device__ __forceinline__ void pair_tile_coords(int tile, const TcParams& p, int& m0, int& n0) {
  const int per_group = RASTER_GROUP * p.tiles_n;
  const int g = tile / per_group;
  const int first_m = g * RASTER_GROUP;
  const int gsize = min(p.tiles_m - first_m, RASTER_GROUP);
  const int local = tile % per_group;
  m0 = (first_m + local % gsize) * BM;
  n0 = (local / gsize) * BN;
}

// TMEM -> registers for one warp's 32 accumulator rows, `chunks` chunks of
// 32 columns from t_row, each handed to use(c, r); arrives on the
// accumulator-empty barrier `tempty` as soon as the last load has landed.
// (Keeping the next chunk's load in flight while a chunk is stored, and
// staging chunks through shared memory for row-contiguous stores, were both
// timed on GB300 and changed nothing.)
template <typename Use>
__device__ __forceinline__ void drain_chunks(uint32_t t_row, int chunks, uint32_t tempty, Use&& use) {
#pragma unroll 1
  for (int c = 0; c < chunks; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + c * 32, r);
    tc_wait_ld();
    if (c == chunks - 1) {
      tc_fence_before();
      mbar_arrive_remote(tempty);
    }
    use(c, r);
  }
}

// Stream-K piece end in the epilogue of one warp (32 rows of one CTA's 128):
// a contributor leaves its rows of the partial tile in its workspace slot and
// raises its flag; the finisher waits (bounded) for the other pairs' flags of
// the same rows, adds their parts to its own in pair order (fixed by the
// shape, so every call gives the same bits), stores C through the usual
// epilogue and lowers the flags.  A warp's part is laid out chunk by chunk
// (32 columns = 8 float4 per row), each float4 of the 32 rows contiguous, so
// every warp access is 512 contiguous bytes.  t_row: this warp's accumulator
// row in TMEM; tempty: the accumulator-empty barrier to arrive on once TMEM
// is read.  Returns false after a bounded wait ran out.
constexpr int kSkMaxWorkers = 16;   // pairs meeting in one tile (at most 5 in practice)
template <int BN, bool OUT_BF16>
__device__ __forceinline__ bool sk_piece_end(const TcParams& p, long long u, int pair_id,
                                             uint32_t rank, int quarter, int lane, long long m,
                                             int n0, uint32_t t_row, uint32_t tempty,
                                             volatile int* abort_flag) {
  const GemmArgs& a = p.a;
  const long long U = p.sk_units;
  const int G = p.sk_pairs;
  const long long T0 = u - u % p.k_tiles, T1 = T0 + p.k_tiles;
  int cfirst, clast, fin;
  sk_tile_workers(T0, T1, U, G, &cfirst, &clast, &fin);
  auto slot_of = [&](int c) {
    return c * 2 + (int)(T0 / p.k_tiles - sk_begin(c, U, G) / p.k_tiles);
  };
  const int flag_idx = (int)rank * 4 + quarter;
  // this warp's block of a slot: 32 rows x BN floats
  auto block = [&](int c) {
    return reinterpret_cast<float4*>(p.sk_partials + (size_t)slot_of(c) * (BM * BN) +
                                     (size_t)flag_idx * (32 * BN));
  };
  if (pair_id != fin) {
    // ------------------------------------------------ contributor
    float4* dst = block(pair_id);
    drain_chunks(t_row, BN / 32, tempty, [&](int c, uint32_t (&r)[32]) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[(c * 8 + q) * 32 + lane] =
            make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                        __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
    });
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_u32(p.sk_flags + slot_of(pair_id) * 8 + flag_idx, 1u);
    return true;
  }
  // -------------------------------------------------- finisher
  bool ok = clast - cfirst < kSkMaxWorkers;
  if (lane == 0 && ok) {
    for (int c = cfirst; ok && c <= clast; ++c) {
      if (c == pair_id) continue;
      const unsigned* flag = p.sk_flags + slot_of(c) * 8 + flag_idx;
      if (ld_acquire_u32(flag) != 0u) continue;
      const uint64_t t0 = globaltimer_ns();
      while (true) {
        bool got = false;
#pragma unroll 1
        for (int i = 0; i < 32 && !got; ++i) got = ld_acquire_u32(flag) != 0u;
        if (got) break;
        if (*abort_flag || globaltimer_ns() - t0 > a.timeout_ns) {
          ok = false;
          break;
        }
      }
    }
  }
  if (lane == 0 && !ok) {
    if (!*abort_flag) report_status(a.status, 5, kSiteTc2StreamK);
    *abort_flag = 1;
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (!ok) {
    // TMEM is still handed back, so the MMA issuer's own wait is not the
    // one that runs out
    tc_fence_before();
    mbar_arrive_remote(tempty);
    return false;
  }
  __syncwarp();
  __threadfence();
  // the other parts in pair order: the j-th is pair cfirst + j, skipping this one
  const int n_src = clast - cfirst;
  auto src_of = [&](int j) -> const float4* {
    const int c = cfirst + j;
    return block(c >= pair_id ? c + 1 : c);
  };
  drain_chunks(t_row, BN / 32, tempty, [&](int c, uint32_t (&r)[32]) {
    // two parts' loads in flight at a time (L2 loads: other SMs wrote them),
    // added in order after this pair's own part
#pragma unroll 1
    for (int j = 0; j < n_src; j += 2) {
      const bool two = j + 1 < n_src;
      const float4* s0 = src_of(j) + c * 8 * 32 + lane;
      const float4* s1 = two ? src_of(j + 1) + c * 8 * 32 + lane : s0;
      float4 v0[8], v1[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v0[q] = __ldcg(s0 + q * 32);
        v1[q] = __ldcg(s1 + q * 32);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        r[4 * q] = __float_as_uint(__uint_as_float(r[4 * q]) + v0[q].x);
        r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + v0[q].y);
        r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + v0[q].z);
        r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + v0[q].w);
      }
      if (two) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          r[4 * q] = __float_as_uint(__uint_as_float(r[4 * q]) + v1[q].x);
          r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + v1[q].y);
          r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + v1[q].z);
          r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + v1[q].w);
        }
      }
    }
    if (m < a.M && n0 + c * 32 < a.N) store_row32<OUT_BF16>(p, m, (long long)n0 + c * 32, r);
  });
  __syncwarp();
  if (lane == 0) {
    for (int c = cfirst; c <= clast; ++c)
      if (c != pair_id) p.sk_flags[slot_of(c) * 8 + flag_idx] = 0u;   // ready for the next call
  }
  return true;
}

// mapB2 is read only by the SwiGLU variant (the up-projection).
// SK: the tiles past the whole waves run stream-K (bf16 and FP8 instances of
// the 256-wide tile; the plain instances have no trace of it).
template <int BN, bool OUT_BF16, bool SW, bool F8, bool SK = false>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_bf16_tc2_kernel(const __grid_constant__ CUtensorMap mapA,
                         const __grid_constant__ CUtensorMap mapB,
                         const __grid_constant__ CUtensorMap mapB2, const TcParams p) {
  static_assert(!SW || (BN == 256 && OUT_BF16 && !F8), "SwiGLU runs on the 256-wide bf16 instance");
  static_assert(!SK || (BN == 256 && !SW), "stream-K runs on the 256-wide plain and FP8 instances");
  constexpr int OUT_BN = SW ? BN / 2 : BN;  // C columns per tile
  using Cfg = PairCfg<BN, F8>;
  using G = Geom<F8>;
  constexpr int BK = G::BK;
  constexpr int A_STAGE_BYTES = G::A_STAGE_BYTES;
  constexpr int B_BOX_BYTES = G::B_BOX_BYTES;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int STAGE_BYTES = Cfg::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  // Same offsets in both CTAs: the paired MMA reads A and B at the
  // descriptor's address in each CTA of the pair.
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar_base = base + STAGES * STAGE_BYTES;
  uint8_t* bar_ptr = base_ptr + STAGES * STAGE_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * STAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_ptr + 8 * (2 * STAGES + 5) + 8);
  const uint32_t stall_bar = bar_base + 8u * (2 * STAGES + 7);  // test hook: nothing arrives
  static_assert(8 * (2 * STAGES + 8) <= BAR_BYTES, "barrier area");
  auto a_tile = [&](int s) { return base + s * STAGE_BYTES; };
  auto b_tile = [&](int s) { return base + s * STAGE_BYTES + A_STAGE_BYTES; };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const GemmArgs& a = p.a;
  const uint32_t rank = cluster_ctarank() & 1u;  // clusters hold exactly one pair
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  // this pair's work items: whole tiles, then at most one half-width item
  // or (SK) the pieces of its stream-K range: units [sk_b, sk_e) of the
  // tail, in tile sk_t0 and, past its end, in the next tile
  const int n_dp = pair_id < p.dp_tiles ? (p.dp_tiles - pair_id + num_pairs - 1) / num_pairs : 0;
  long long sk_b = 0, sk_e = 0;
  int sk_t0 = 0, sk_pieces = 0;
  if constexpr (SK) {
    if (pair_id < p.sk_pairs) {
      sk_b = sk_begin(pair_id, p.sk_units, p.sk_pairs);
      sk_e = sk_begin(pair_id + 1, p.sk_units, p.sk_pairs);
      sk_t0 = (int)(sk_b / p.k_tiles);
      sk_pieces = sk_e <= sk_b ? 0 : sk_e > (long long)(sk_t0 + 1) * p.k_tiles ? 2 : 1;
    }
  }
  const int n_items = n_dp + (SK ? sk_pieces : (pair_id < p.half_tiles ? 1 : 0));
  // K-steps [k_lo, k_hi) of item i; u: its first unit in the stream-K run
  auto item_k = [&](int i, int& k_lo, int& k_hi, long long& u) {
    k_lo = 0;
    k_hi = p.k_tiles;
    u = 0;
    if constexpr (SK) {
      if (i >= n_dp) {
        const long long t0_unit = (long long)sk_t0 * p.k_tiles;
        if (i == n_dp) {
          u = sk_b;
          k_lo = (int)(sk_b - t0_unit);
          k_hi = (int)((sk_e < t0_unit + p.k_tiles ? sk_e : t0_unit + p.k_tiles) - t0_unit);
        } else {
          u = t0_unit + p.k_tiles;
          k_hi = (int)(sk_e - u);
        }
      }
    }
  };
  auto item = [&](int i, int& m0, int& n0, int& bn) {
    if (i < n_dp) {
      pair_tile_coords<OUT_BN>(pair_id + i * num_pairs, p, m0, n0);
      bn = BN;
    } else if constexpr (SK) {
      pair_tile_coords<OUT_BN>(p.dp_tiles + sk_t0 + (i - n_dp), p, m0, n0);
      bn = BN;
    } else {
      pair_tile_coords<OUT_BN>(p.dp_tiles + pair_id / 2, p, m0, n0);
      bn = BN / 2;
      n0 += (pair_id & 1) * (BN / 2);
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * NUM_EPI_WARPS * 32);
    }
    mbar_init(drain_bar, 1);
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one_sync()) {
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapB);
      if (SW) tma_prefetch_desc(&mapB2);
      uint32_t issued = 0, issued_par = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_items; ++i) {
        int m0, n0, bn, k_lo, k_hi;
        long long u;
        item(i, m0, n0, bn);
        item_k(i, k_lo, k_hi, u);
        const int a_row = m0 + (int)rank * BM_CTA;
        const int b_col = n0 + (int)rank * (SW ? OUT_BN / 2 : bn / 2);
        const int b_boxes = bn / 2 / G::BOX_N;
        const uint32_t tx_bytes = 2u * (A_STAGE_BYTES + b_boxes * B_BOX_BYTES);
        for (int kt = k_lo; kt < k_hi; ++kt) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, a.timeout_ns, abort_flag)) {
            if (!*abort_flag) report_status(a.status, 5, kSiteTc2Producer);
            *abort_flag = 1;
            ok = false;
            break;
          }
          // both CTAs' copies of this stage complete on the leader's barrier
          const uint32_t lead_full = map_to_rank(full_bar(stage), 0);
          if (leader) mbar_arrive_expect_tx(full_bar(stage), tx_bytes);
          tma_load_2d_pair(a_tile(stage), &mapA, lead_full, kt * BK, a_row);
          for (int j = 0; j < b_boxes; ++j)
            tma_load_2d_pair(b_tile(stage) + j * B_BOX_BYTES, (SW && j == 1) ? &mapB2 : &mapB,
                             lead_full, SW ? b_col : b_col + j * G::BOX_N, kt * BK);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        if (leader) {
          for (int s = 0; s < STAGES; ++s)
            if (((issued >> s) & 1u) &&
                !mbar_wait(full_bar(s), (issued_par >> s) & 1u, kDrainWaitNs, nullptr))
              report_status(a.status, 5, kSiteTc2Drain);
        }
        // the peer's copies complete on a barrier this CTA cannot wait on:
        // give them a bounded grace period before shared memory is released
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kDrainGraceNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (leader) {
      if (elect_one_sync()) {
        const uint32_t idesc_full =
            F8 ? idesc_f8_f32(BM, BN, (uint32_t)a.fmt_a, (uint32_t)a.fmt_b, /*A K-major*/ 0, /*B MN-major*/ 1)
               : idesc_bf16_f32(BM, BN, /*A K-major*/ 0, /*B MN-major*/ 1);
        const uint32_t idesc_half = idesc_bf16_f32(BM, BN / 2, 0, 1);  // bf16 only
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true, issued_any = false;
        if (a.stall && pair_id == 0 && !mbar_wait(stall_bar, 0, a.timeout_ns / 4, abort_flag)) {
          // test hook: this wait runs out; the pair takes its abort path
          if (!*abort_flag) report_status(a.status, 5, kSiteTc2Mma);
          *abort_flag = 1;
          ok = false;
        }
        for (int i = 0; ok && i < n_items; ++i) {
          // stream-K pieces are whole-width tiles; only the half-width tail
          // (bf16 instances without SK; never FP8) uses the 128-wide descriptor
          const uint32_t idesc = (SK || F8 || i < n_dp) ? idesc_full : idesc_half;
          if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, a.timeout_ns, abort_flag)) {
            if (!*abort_flag) report_status(a.status, 5, kSiteTc2Mma);
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
          int k_lo, k_hi;
          long long u;
          item_k(i, k_lo, k_hi, u);
          for (int kt = k_lo; kt < k_hi; ++kt) {
            if (!mbar_wait(full_bar(stage), phase, a.timeout_ns, abort_flag)) {
              if (!*abort_flag) report_status(a.status, 5, kSiteTc2Mma);
              *abort_flag = 1;
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < BK / G::UMMA_K; ++kk) {
              const uint64_t adesc = smem_desc_sw128(a_tile(stage) + kk * G::A_KSTEP, 16, 1024);
              const uint64_t bdesc =
                  smem_desc_sw128(b_tile(stage) + kk * G::B_KSTEP, B_BOX_BYTES, 1024);
              const uint32_t accumulate = (kt != k_lo || kk != 0) ? 1u : 0u;
              if constexpr (F8)
                tc_mma_f8_pair(d_tmem, adesc, bdesc, idesc, accumulate);
              else
                tc_mma_f16_pair(d_tmem, adesc, bdesc, idesc, accumulate);
            }
            issued_any = true;
            tc_commit_pair_mc(empty_bar(stage), kBothCtas);  // frees the stage in both CTAs
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_pair_mc(tfull_bar(acc), kBothCtas);  // both halves of D are ready
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        if (*abort_flag && issued_any) {
          tc_commit_pair_mc(drain_bar, 0x1);
          if (!mbar_wait(drain_bar, 0, kDrainWaitNs, nullptr)) report_status(a.status, 5, kSiteTc2Drain);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp % 4;
    const uint32_t lead_tempty0 = map_to_rank(tempty_bar(0), 0);
    const uint32_t lead_tempty1 = map_to_rank(tempty_bar(1), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int i = 0; i < n_items; ++i) {
      int m0, n0, bn;
      item(i, m0, n0, bn);
      // warp-uniform (the tcgen05.ld below is warp-wide)
      if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), acc_phase, a.timeout_ns, abort_flag))) {
        if (!*abort_flag) report_status(a.status, 5, kSiteTc2Epilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const long long m = (long long)m0 + rank * BM_CTA + quarter * 32 + lane;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (SK && i >= n_dp) {
        // ------------------------------------------ stream-K piece end
        int k_lo, k_hi;
        long long u;
        item_k(i, k_lo, k_hi, u);
        if (!sk_piece_end<BN, OUT_BF16>(p, u, pair_id, rank, quarter, lane, m, n0, t_row,
                                        acc == 0 ? lead_tempty0 : lead_tempty1, abort_flag))
          break;
      } else if constexpr (SW) {
#pragma unroll 1
        for (int c = 0; c < OUT_BN / 32; ++c) {
          // output columns n0 + 32c .. +32: gate at accumulator column
          // 128*(c/2) + 32*(c%2), the up projection 64 columns further on
          const uint32_t g_col = (uint32_t)(128 * (c / 2) + 32 * (c % 2));
          uint32_t r[32], u[32];
          tmem_ld_32x32b_x32(t_row + g_col, r);
          tmem_ld_32x32b_x32(t_row + g_col + 64, u);
          tc_wait_ld();
          if (c == OUT_BN / 32 - 1) {
            tc_fence_before();
            mbar_arrive_remote(acc == 0 ? lead_tempty0 : lead_tempty1);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j)
            r[j] = __float_as_uint(swiglu_combine(__uint_as_float(r[j]), __uint_as_float(u[j])));
          if (m < a.M && n0 + c * 32 < a.N) store_row32<OUT_BF16>(p, m, (long long)n0 + c * 32, r);
        }
      } else {
        drain_chunks(t_row, bn / 32, acc == 0 ? lead_tempty0 : lead_tempty1,
                     [&](int c, uint32_t (&r)[32]) {
                       if (m < a.M && n0 + c * 32 < a.N)
                         store_row32<OUT_BF16>(p, m, (long long)n0 + c * 32, r);
                     });
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  cluster_sync();  // both CTAs are done with the pair's TMEM and barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

struct PairLaunchInfo {
  std::atomic<bool> ready{false};   // published after max_clusters is set
  int max_clusters = 0;
};

template <int BN, bool OUT_BF16, bool SW, bool F8 = false>
int launch_pair_impl(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                     const CUtensorMap* mapB2, int num_sms, cudaStream_t s, int* schedule) {
  constexpr int OUT_BN = SW ? BN / 2 : BN;
  using Cfg = PairCfg<BN, F8>;
  constexpr int BK = Geom<F8>::BK;
  static PairLaunchInfo info[64];
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kernel = gemm_bf16_tc2_kernel<BN, OUT_BF16, SW, F8>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!info[dev].ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(mu);
    if (!info[dev].ready.load(std::memory_order_relaxed)) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Cfg::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      // clusters that can be resident at once (GPCs with an odd number of
      // free SMs leave one idle), so the persistent grid never has a tail
      int n = 0;
      cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
      e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
      if (e != cudaSuccess) return e;
      info[dev].max_clusters = n > 0 ? n : 1;
      info[dev].ready.store(true, std::memory_order_release);
    }
  }
  TcParams p;
  p.a = a;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = (a.N + OUT_BN - 1) / OUT_BN;
  const long long tiles = (long long)p.tiles_m * p.tiles_n;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.num_tiles = (int)tiles;
  p.k_tiles = (a.K + BK - 1) / BK;
  const int out_bytes = OUT_BF16 ? 2 : 4;
  p.c_vec = ((reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && ((a.ldc * out_bytes) % 16) == 0) ? 1 : 0;
  const int pairs = info[dev].max_clusters;
  const long long rem = tiles % pairs;
  // the tiles past the last whole wave: whole (0), as half-width tiles (1)
  // or stream-K over the pairs (2), as the tail model or the hook says
  int tail = 0, sk_pairs = 0;
  const int mode = split_tiles_mode();
  if (!SW && BN == 256 && mode != 0 && rem > 0) {
    const bool half_ok = !F8 && 2 * rem <= pairs;
    sk_pairs = plan::tc_sk_pairs(rem, p.k_tiles, pairs);
    if (mode == 2) tail = sk_pairs > 0 ? 2 : 0;
    else if (mode == 3) tail = half_ok ? 1 : 0;
    else tail = plan::tc_tail(rem, pairs, half_ok, sk_pairs);
  }
  int clusters;
  if constexpr (!SW && BN == 256) {
    if (tail == 2) {
      static std::atomic<uint64_t> smem_sk{0};
      auto sk_kernel = gemm_bf16_tc2_kernel<BN, OUT_BF16, SW, F8, true>;
      cudaError_t e = set_smem_once(smem_sk, sk_kernel, Cfg::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      float* partials = nullptr;
      unsigned* flags = nullptr;
      size_t slot_floats = 0, slot_flags = 0;
      if ((e = stream_k_slot(num_sms, &partials, &flags, &slot_floats, &slot_flags)) != cudaSuccess)
        return e;
      if ((size_t)sk_pairs * 2 * BM * BN > slot_floats || (size_t)sk_pairs * 2 * 8 > slot_flags)
        return cudaErrorInvalidValue;
      p.dp_tiles = (int)(tiles - rem);
      p.half_tiles = 0;
      p.sk_pairs = sk_pairs;
      p.sk_units = rem * p.k_tiles;
      p.sk_partials = partials;
      p.sk_flags = flags;
      *schedule = 6;
      cfg.gridDim = dim3(2 * pairs, 1, 1);
      e = cudaLaunchKernelEx(&cfg, sk_kernel, *mapA, *mapB, *mapB, p);
      if (e != cudaSuccess) return e;
      return cudaGetLastError();
    }
  }
  if (tail == 1) {
    p.dp_tiles = (int)(tiles - rem);
    p.half_tiles = (int)(2 * rem);
    clusters = pairs;
    *schedule = 4;
  } else {
    p.dp_tiles = p.num_tiles;
    p.half_tiles = 0;
    clusters = (int)(tiles < pairs ? tiles : pairs);
    *schedule = 2;
  }
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, *mapA, *mapB, SW ? *mapB2 : *mapB, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int launch_bf16_tc_pair(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB, int bn,
                        int num_sms, cudaStream_t s, int* schedule) {
  const bool bf16 = a.out == Elem::BF16;
  if (bn == 256)
    return bf16 ? launch_pair_impl<256, true, false>(a, mapA, mapB, nullptr, num_sms, s, schedule)
                : launch_pair_impl<256, false, false>(a, mapA, mapB, nullptr, num_sms, s, schedule);
  if (bn == 128)
    return bf16 ? launch_pair_impl<128, true, false>(a, mapA, mapB, nullptr, num_sms, s, schedule)
                : launch_pair_impl<128, false, false>(a, mapA, mapB, nullptr, num_sms, s, schedule);
  return cudaErrorInvalidValue;
}

int launch_fp8_tc_pair(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                       int num_sms, cudaStream_t s, int* schedule) {
  if (a.in != Elem::FP8 || a.swiglu) return cudaErrorInvalidValue;
  return a.out == Elem::BF16
             ? launch_pair_impl<256, true, false, true>(a, mapA, mapB, nullptr, num_sms, s, schedule)
             : launch_pair_impl<256, false, false, true>(a, mapA, mapB, nullptr, num_sms, s, schedule);
}

int launch_bf16_swiglu_pair(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                            const CUtensorMap* mapB2, int num_sms, cudaStream_t s) {
  if (!a.swiglu || a.out != Elem::BF16 || mapB2 == nullptr) return cudaErrorInvalidValue;
  int schedule = 0;
  return launch_pair_impl<256, true, true>(a, mapA, mapB, mapB2, num_sms, s, &schedule);
}

}  // namespace g3
