// BF16 GEMM on the 5th-generation tensor cores: C = alpha*A*B + beta*C with
// bf16 A (M x K, row-major) and B (K x N, row-major), fp32 accumulation, bf16
// or fp32 C.
//
// The structure is the Blackwell pipeline of "Kernel 性能从何而来":
//   * section "优化阶梯": tiles move by TMA, the tensor-core math is
//     tcgen05.mma with the accumulator in TMEM, roles are warp-specialised;
//   * section "通过重叠执行减少硬件空闲": load tile k+1, compute tile k and
//     store tile k-1 at the same time, handed over by mbarriers.  Here a
//     4-stage shared-memory ring overlaps TMA with MMA, and two TMEM
//     accumulators let the epilogue of one C tile run under the main loop of
//     the next;
//   * section "SM 占用率与资源压力": one CTA per SM holding ~193 KB of staging
//     and all 512 TMEM columns, trading occupancy for deep staging.
// The per-stage tile is 128 x 256 with B_K = 64, a per-stage A/B intensity of
// 2*128*256*64 / (2*(128*64 + 64*256)) = 85 FLOP/byte (section
// "优化 Memory-Bound Kernel", blocking), against 8 and 32 for the 16x16 and
// 64x64 examples there.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM allocator and
// MMA issuer (one elected thread), warps 2-5 = epilogue (TMEM -> registers ->
// alpha/beta in fp32 -> C).  A is K-major in shared memory (one 128-byte
// swizzle atom spans the 64 K of a stage); B is N-major (row-major B has N
// contiguous), loaded as four 64-column boxes that form four MN atoms.
//
// The persistent grid has one CTA per SM and walks C tiles in a grouped
// raster.  Every wait is bounded: a wait that runs out records a timeout in
// the device status word and every role leaves its loop, after which the CTA
// lets its copies and MMAs land and frees TMEM before returning.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "plan.h"
#include "ptx.cuh"
#include "tc_epilogue.cuh"

namespace g3 {
namespace {

constexpr int BM = kTcBM, BK = kTcBK;
constexpr int UMMA_K = 16;
constexpr int A_STAGE_BYTES = BM * BK * 2;                // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;                  // 8 KB (64 n x 64 k)
constexpr int TMEM_COLS = 512;                            // two accumulators of up to 256 columns
constexpr int NUM_EPI_WARPS = 4;
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_LIMIT = 232448;                        // opt-in dynamic shared memory per CTA
constexpr int RASTER_GROUP = 16;

// Tile geometry for a C tile of BM x BN.  B is loaded as ceil(BN/64) boxes of
// 64 columns; the MMA reads BN of them.
template <int BN>
struct TileCfg {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "tcgen05 N for M=128, 32-column epilogue");
  static constexpr int B_BOXES = (BN + 63) / 64;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_BOXES * B_BOX_BYTES;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - BAR_BYTES - 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
  static_assert(2 * BN <= TMEM_COLS, "two accumulators must fit in TMEM");
};

template <int BN>
__device__ __forceinline__ void tile_coords(int tile, const TcParams& p, int& m0, int& n0) {
  const int per_group = RASTER_GROUP * p.tiles_n;
  const int g = tile / per_group;
  const int first_m = g * RASTER_GROUP;
  const int gsize = min(p.tiles_m - first_m, RASTER_GROUP);
  const int local = tile % per_group;
  m0 = (first_m + local % gsize) * BM;
  n0 = (local / gsize) * BN;
}

template <int BN, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB, const TcParams p) {
  using Cfg = TileCfg<BN>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int STAGE_BYTES = Cfg::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-byte alignment
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar_base = base + STAGES * STAGE_BYTES;
  uint8_t* bar_ptr = base_ptr + STAGES * STAGE_BYTES;
  // barrier layout: full[S], empty[S], tmem_full[2], tmem_empty[2], drain
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * STAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_ptr + 8 * (2 * STAGES + 5) + 8);
  auto a_tile = [&](int s) { return base + s * STAGE_BYTES; };
  auto b_tile = [&](int s) { return base + s * STAGE_BYTES + A_STAGE_BYTES; };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const GemmArgs& a = p.a;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), NUM_EPI_WARPS * 32);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one_sync()) {
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapB);
      // bit s of `issued`: slot s has had a copy issued; bit s of
      // `issued_par`: the phase parity of its latest copy
      uint32_t issued = 0, issued_par = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        int m0, n0;
        tile_coords<BN>(tile, p, m0, n0);
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, a.timeout_ns, abort_flag)) {
            if (!*abort_flag) report_status(a.status, 5, kSiteTcProducer);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
          tma_load_2d(a_tile(stage), &mapA, full_bar(stage), kt * BK, m0);
#pragma unroll
          for (int j = 0; j < Cfg::B_BOXES; ++j)
            tma_load_2d(b_tile(stage) + j * B_BOX_BYTES, &mapB, full_bar(stage), n0 + j * 64,
                        kt * BK);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < STAGES; ++s)
          if (((issued >> s) & 1u) &&
              !mbar_wait(full_bar(s), (issued_par >> s) & 1u, kDrainWaitNs, nullptr))
            report_status(a.status, 5, kSiteTcDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_sync()) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, /*A K-major*/ 0, /*B MN-major*/ 1);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued_any = false;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, a.timeout_ns, abort_flag)) {
          if (!*abort_flag) report_status(a.status, 5, kSiteTcMma);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(full_bar(stage), phase, a.timeout_ns, abort_flag)) {
            if (!*abort_flag) report_status(a.status, 5, kSiteTcMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            // A: K-major, the 16-element K step moves 32 bytes inside the atom.
            const uint64_t adesc = smem_desc_sw128(a_tile(stage) + kk * UMMA_K * 2, 16, 1024);
            // B: N-major, the K step moves 16 rows of 128 bytes; atoms of 64
            // columns are B_BOX_BYTES apart, 8-row groups 1024 bytes apart.
            const uint64_t bdesc =
                smem_desc_sw128(b_tile(stage) + kk * UMMA_K * 128, B_BOX_BYTES, 1024);
            tc_mma_f16(d_tmem, adesc, bdesc, idesc, (kt | kk) != 0 ? 1u : 0u);
          }
          issued_any = true;
          tc_commit(empty_bar(stage));  // frees the stage once these MMAs have read it
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));  // accumulator ready for the epilogue
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (*abort_flag && issued_any) {
        // all MMAs issued so far must finish before TMEM and shared memory go away
        tc_commit(drain_bar);
        if (!mbar_wait(drain_bar, 0, kDrainWaitNs, nullptr)) report_status(a.status, 5, kSiteTcDrain);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp % 4;  // TMEM lanes [32*quarter, 32*quarter+32) belong to this warp
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      int m0, n0;
      tile_coords<BN>(tile, p, m0, n0);
      // warp-uniform (the tcgen05.ld below is warp-wide)
      if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), acc_phase, a.timeout_ns, abort_flag))) {
        if (!*abort_flag) report_status(a.status, 5, kSiteTcEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const long long m = (long long)m0 + quarter * 32 + lane;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tc_wait_ld();
        if (c == BN / 32 - 1) {
          // accumulator fully read: hand it back before the last stores
          tc_fence_before();
          mbar_arrive(tempty_bar(acc));
        }
        if (m < a.M && n0 + c * 32 < a.N) store_row32<OUT_BF16>(p, m, (long long)n0 + c * 32, r);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int BN, bool OUT_BF16>
int launch_impl(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB, int num_sms,
                cudaStream_t s) {
  using Cfg = TileCfg<BN>;
  static std::atomic<uint64_t> smem_set{0};
  {
    cudaError_t e = set_smem_once(smem_set, gemm_bf16_tc_kernel<BN, OUT_BF16>, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  TcParams p;
  p.a = a;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = (a.N + BN - 1) / BN;
  const long long tiles = (long long)p.tiles_m * p.tiles_n;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.num_tiles = (int)tiles;
  p.k_tiles = (a.K + BK - 1) / BK;
  const int out_bytes = OUT_BF16 ? 2 : 4;
  p.c_vec = ((reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && ((a.ldc * out_bytes) % 16) == 0) ? 1 : 0;
  const int grid = (int)(tiles < num_sms ? tiles : num_sms);
  gemm_bf16_tc_kernel<BN, OUT_BF16><<<grid, THREADS, Cfg::SMEM_BYTES, s>>>(*mapA, *mapB, p);
  return cudaGetLastError();
}

template <bool OUT_BF16>
int launch_bn(int bn, const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
              int num_sms, cudaStream_t s) {
  switch (bn) {
    case 256: return launch_impl<256, OUT_BF16>(a, mapA, mapB, num_sms, s);
    case 224: return launch_impl<224, OUT_BF16>(a, mapA, mapB, num_sms, s);
    case 192: return launch_impl<192, OUT_BF16>(a, mapA, mapB, num_sms, s);
    case 128: return launch_impl<128, OUT_BF16>(a, mapA, mapB, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// The wave models live in plan.h (host arithmetic shared with a CPU test).
int choose_tc_bn(int M, int N, int num_sms) { return plan::tc_bn(M, N, num_sms); }

void choose_tc_config(int M, int N, int num_sms, int* pair, int* bn) {
  plan::tc_config(M, N, num_sms, split_tiles_enabled(), pair, bn);
}

int launch_bf16_tc(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                   int bn, int num_sms, cudaStream_t s) {
  if (a.out == Elem::BF16) return launch_bn<true>(bn, a, mapA, mapB, num_sms, s);
  return launch_bn<false>(bn, a, mapA, mapB, num_sms, s);
}

}  // namespace g3
