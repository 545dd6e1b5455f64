// INT4 weight-only decode GEMM: C = alpha * X * W + beta * C with X bf16
// (M <= 16 rows), W = s[k / G][n] * (q[k][n] - z) given as 4-bit codes, fp32
// accumulation, bf16 or fp32 C.
//
// "CUDA 算子工程 ch.4 内存层级与代价表", section 4.5.3: INT4 dequantisation
// is the memory-bound workload next to the decode GEMM, and the codes move a
// quarter of the bytes of bf16 weights; "Kernel 性能从何而来", section
// "优化 Memory-Bound Kernel": fuse the producer (dequantisation) with its
// consumer (the GEMM) so the bf16 weight never goes to HBM.  Design:
//   * the operands are swapped as in the bf16 decode kernel: 128 columns of W
//     are the MMA's M = 128 rows, the <= 16 activation rows its N = 16;
//   * the codes stream once from HBM into an 8-stage shared-memory ring: a
//     stage is two adjacent 4 KB tiles of codes (128 columns x 128 rows of K,
//     one contiguous bulk copy, so every DRAM access is sequential) plus 4 KB
//     of X by TMA; the ring's size also keeps a third CTA off the SM, so two
//     CTAs' 256 tensor-memory columns are never waited for inside a cluster;
//     a stage is 128 rows deep so that the single MMA thread's fixed cost
//     (barrier waits, commits) is paid once per eight MMAs;
//   * two groups of four dequantisation warps, taking alternate stages, turn
//     each column's 64 codes into the exact bf16 integers q - z (two codes per
//     step: one lop3 makes the magic-number bf16 pair 128 + code, one packed
//     bf16 FMA subtracts 128 + z) and write them, eight columns per store,
//     straight into tensor memory with tcgen05.st, so the weight operand
//     never passes through shared memory (a bf16 tile written and read back
//     there would need more shared-memory bandwidth per SM than the HBM rate
//     leaves); two groups keep two stages' load-convert-store chains in flight;
//   * one thread issues tcgen05.mma with A read from tensor memory, into one
//     of four accumulators per group of G rows of W; the first dequantisation
//     group drains each accumulator, scales it by s[group][n] in fp32 (the
//     scale fetched a group ahead) and adds it to its registers (the weight
//     is never rounded);
//   * K is split over a cluster of S <= 8 CTAs along whole groups; the
//     partials meet over distributed shared memory in rank order, and the
//     alpha/beta epilogue is fused into that reduction.
// The codes are in the tiled layout that gemm_int4_repack writes: tiles of
// 128 columns x 64 rows of K, 4 KB each, column tiles outer and K tiles
// inner; inside a tile column n has 32 bytes = eight little-endian 32-bit
// words, word j the codes of k = 8j + (0,2,4,6,1,3,5,7) in its nibbles 0..7,
// so that bits 0-3 and 16-19 of (word >> 4i) are the codes of k = 8j + 2i
// and 8j + 2i + 1.  Tiles past N or K hold zero codes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>

#include "internal.h"
#include "plan.h"
#include "ptx.cuh"

namespace g3 {
namespace {

constexpr int BN = kW4BN;            // W columns per CTA (MMA M, TMEM lanes)
constexpr int BK = kW4BK;            // K rows per tile of codes (a "chunk")
constexpr int MN = kSkMaxM;          // MMA N: activation rows, zero-padded by TMA
constexpr int UMMA_K = 16;
constexpr int CPS = 2;               // chunks per pipeline stage (128 rows of K)
constexpr int SSTAGES = 8;           // shared-memory ring of codes + X
constexpr int ASTAGES = 3;           // tensor-memory ring of dequantised weights
constexpr int NACC = 4;              // accumulators (groups in flight)
constexpr int CODE_CHUNK_BYTES = BN * BK / 2;            // 4 KB: one tile
constexpr int X_CHUNK_BYTES = MN * BK * 2;               // 2 KB: one TMA box
constexpr int CODE_STAGE_BYTES = CPS * CODE_CHUNK_BYTES; // 8 KB
constexpr int X_STAGE_BYTES = CPS * X_CHUNK_BYTES;       // 4 KB
constexpr int STAGE_BYTES = CODE_STAGE_BYTES + X_STAGE_BYTES;
constexpr int DQ_GROUPS = 2;         // dequantisation warp groups, alternate stages
constexpr int THREADS = 64 + DQ_GROUPS * 128;   // producer, MMA, 4 warps per group
constexpr int TMEM_COLS = 256;
constexpr int A_COLS = CPS * BK / 2; // TMEM columns per dequantised stage
constexpr int ACC_COL0 = ASTAGES * A_COLS;               // 192
constexpr int MAX_SPLIT = 8;
constexpr int PARTIAL_BYTES = MN * BN * 4;               // 8 KB
constexpr int BAR_BYTES = 512;
constexpr int SMEM_BYTES = SSTAGES * STAGE_BYTES + BAR_BYTES + 1024;
static_assert(ACC_COL0 + NACC * MN <= TMEM_COLS, "tensor memory budget");
static_assert(PARTIAL_BYTES <= SSTAGES * STAGE_BYTES, "partial tile aliases the ring");
static_assert(X_CHUNK_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "1024-byte stage alignment");
// at most two CTAs per SM (shared memory 228 KB, 1 KB reserved per CTA), so
// their 2 x 256 tensor-memory columns are always free at allocation
static_assert(3 * (SMEM_BYTES + 1024) > 228 * 1024, "a third CTA must not fit");

struct W4Params {
  GemmArgs a;                // A = X (M x K bf16), C
  const uint8_t* qk;         // tiled codes
  const __nv_bfloat16* scales;
  long long lds;
  int group, zero;
  int k_tiles;               // chunks of 64 rows over all of K
  int stages_per_group;      // chunks per group: G / 64, or k_tiles when one group spans K
  int groups;                // groups over all of K
  int split;                 // CTAs per cluster along K
};

// (a & mask) | magic in one instruction (lop3)
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
  return d;
}
// a * 1 + c on bf16 pairs: one packed FMA (exact here: the operands are
// integers below 256)
__device__ __forceinline__ uint32_t fma1_bf16x2(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0x3F803F80u), "r"(c));
  return d;
}
// 8 consecutive 32-bit columns of this thread's TMEM lane; eight registers
// per store keep the dequantised words where the arithmetic left them
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]) : "memory");
}

template <bool OUT_BF16>
__device__ __forceinline__ void store_out(const GemmArgs& a, int m, long long n, float v) {
  const long long off = (long long)m * a.ldc + n;
  if (OUT_BF16)
    static_cast<__nv_bfloat16*>(a.C)[off] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(a.C)[off] = v;
}
template <bool OUT_BF16>
__device__ __forceinline__ float load_out(const GemmArgs& a, int m, long long n) {
  const long long off = (long long)m * a.ldc + n;
  if (OUT_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(a.C)[off]);
  return static_cast<const float*>(a.C)[off];
}

// ring position: slot and phase parity, advanced without division
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

template <bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 2)
    gemm_w4_decode_kernel(const __grid_constant__ CUtensorMap mapX, const W4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar_base = base + SSTAGES * STAGE_BYTES;
  uint8_t* bar_ptr = base_ptr + SSTAGES * STAGE_BYTES;
  auto code_full = [&](int s) { return bar_base + 8u * s; };
  auto code_empty = [&](int s) { return bar_base + 8u * (SSTAGES + s); };
  auto a_full = [&](int s) { return bar_base + 8u * (2 * SSTAGES + s); };
  auto a_empty = [&](int s) { return bar_base + 8u * (2 * SSTAGES + ASTAGES + s); };
  auto acc_full = [&](int r) { return bar_base + 8u * (2 * SSTAGES + 2 * ASTAGES + r); };
  auto acc_empty = [&](int r) { return bar_base + 8u * (2 * SSTAGES + 2 * ASTAGES + NACC + r); };
  constexpr int NBARS = 2 * SSTAGES + 2 * ASTAGES + 2 * NACC + 1;
  static_assert(NBARS * 8 + 16 <= BAR_BYTES, "barrier area");
  const uint32_t drain_bar = bar_base + 8u * (NBARS - 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_ptr + 8 * NBARS + 8);
  auto x_tile = [&](int s) { return base + s * STAGE_BYTES; };
  auto code_tile = [&](int s) { return base + s * STAGE_BYTES + X_STAGE_BYTES; };
  float* partial = reinterpret_cast<float*>(base_ptr);  // [MN][BN], valid after the main loop

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const GemmArgs& a = p.a;
  const int rank = (int)cluster_ctarank();
  const int n0 = blockIdx.y * BN;
  // whole groups per rank, then their chunks and stages
  const int g_begin = (int)((long long)p.groups * rank / p.split);
  const int g_end = (int)((long long)p.groups * (rank + 1) / p.split);
  const int spg = p.stages_per_group;   // chunks per group
  const int kt_begin = min(g_begin * spg, p.k_tiles);
  const int kt_end = min(g_end * spg, p.k_tiles);
  const int my_kt = kt_end - kt_begin;                 // chunks
  const int my_stages = (my_kt + CPS - 1) / CPS;
  const int my_groups = (my_kt + spg - 1) / spg;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SSTAGES; ++s) {
      mbar_init(code_full(s), 1);
      mbar_init(code_empty(s), 4 + 1);  // four dequantisation warps and the MMA's reads of X
    }
    for (int s = 0; s < ASTAGES; ++s) {
      mbar_init(a_full(s), 4);
      mbar_init(a_empty(s), 1);
    }
    for (int r = 0; r < NACC; ++r) {
      mbar_init(acc_full(r), 1);
      mbar_init(acc_empty(r), 4);
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
  if (warp == 0 && lane == 0 && my_kt > 0) {
    // While the previous kernel on the stream finishes, pull this CTA's
    // first stages of codes into L2 (a prefetch only: the copies after the
    // wait read whatever memory holds then, through L2).
    const uint8_t* tiles = p.qk + ((size_t)blockIdx.y * p.k_tiles + kt_begin) * CODE_CHUNK_BYTES;
    const int pre = my_kt < CPS * SSTAGES ? my_kt : CPS * SSTAGES;
    bulk_prefetch_l2(tiles, (uint32_t)pre * CODE_CHUNK_BYTES);
  }
  griddep_wait();  // inputs may come from the previous kernel on the stream

  float acc[MN];
#pragma unroll
  for (int m = 0; m < MN; ++m) acc[m] = 0.f;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one_sync() && my_kt > 0) {
      tma_prefetch_desc(&mapX);
      const uint64_t stream_policy = l2_policy_evict_first();
      const uint8_t* tiles = p.qk + ((size_t)blockIdx.y * p.k_tiles + kt_begin) * CODE_CHUNK_BYTES;
      uint32_t issued = 0, issued_par = 0;
      Ring rs;
      for (int i = 0; i < my_stages; ++i) {
        if (!mbar_wait(code_empty(rs.slot), rs.phase ^ 1u, a.timeout_ns, abort_flag)) {
          if (!*abort_flag) report_status(a.status, 5, kSiteW4Producer);
          *abort_flag = 1;
          break;
        }
        const int c0 = CPS * i;                       // first chunk (local)
        const int nc = min(CPS, my_kt - c0);
        mbar_arrive_expect_tx(code_full(rs.slot), (uint32_t)nc * (CODE_CHUNK_BYTES + X_CHUNK_BYTES));
        // the stage's tiles are adjacent in memory: one contiguous copy
        bulk_load_g2s_hint(code_tile(rs.slot), tiles + (size_t)c0 * CODE_CHUNK_BYTES,
                           (uint32_t)nc * CODE_CHUNK_BYTES, code_full(rs.slot), stream_policy);
        for (int c = 0; c < nc; ++c)
          tma_load_2d(x_tile(rs.slot) + c * X_CHUNK_BYTES, &mapX, code_full(rs.slot),
                      (kt_begin + c0 + c) * BK, 0);
        issued |= 1u << rs.slot;
        issued_par = (issued_par & ~(1u << rs.slot)) | (rs.phase << rs.slot);
        rs.advance(SSTAGES);
      }
      if (*abort_flag) {
        for (int s = 0; s < SSTAGES; ++s)
          if (((issued >> s) & 1u) &&
              !mbar_wait(code_full(s), (issued_par >> s) & 1u, kDrainWaitNs, nullptr))
            report_status(a.status, 5, kSiteW4Drain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_sync() && my_kt > 0) {
      // D^T (128 x 16) += Wq^T (128 x 16, tensor memory) * X^T (16 x 16, K-major)
      constexpr uint32_t idesc = idesc_bf16_f32(BN, MN, 0, 0);
      // The thread shares its scheduler with dequantisation warps, so the loop
      // is kept lean: per stage two waits, one base descriptor and TMEM
      // address with constant offsets, the chunks unrolled, and the group
      // bookkeeping only where a group starts or ends.
      bool ok = true, issued_any = false;
      Ring rs, ra, rr;     // shared-memory stage, tensor-memory stage, accumulator
      int pos = 0;         // chunks of the current group already accumulated
      for (int i = 0; ok && i < my_stages; ++i) {
        if (!mbar_wait(a_full(ra.slot), ra.phase, a.timeout_ns, abort_flag) ||
            !mbar_wait(code_full(rs.slot), rs.phase, a.timeout_ns, abort_flag)) {
          if (!*abort_flag) report_status(a.status, 5, kSiteW4Mma);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int nc = min(CPS, my_kt - CPS * i);
        const uint32_t a0 = tmem_base + (uint32_t)(ra.slot * A_COLS);
        const uint64_t b0 = smem_desc_sw128(x_tile(rs.slot), 16, 1024);
#pragma unroll
        for (int c = 0; c < CPS; ++c) {
          if (c < nc) {
            if (pos == 0) {
              if (!mbar_wait(acc_empty(rr.slot), rr.phase ^ 1u, a.timeout_ns, abort_flag)) {
                if (!*abort_flag) report_status(a.status, 5, kSiteW4Mma);
                *abort_flag = 1;
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d_tmem = tmem_base + (uint32_t)(ACC_COL0 + rr.slot * MN);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              tc_mma_f16_tmem_a(d_tmem, a0 + (uint32_t)(c * (BK / 2) + kk * (UMMA_K / 2)),
                                b0 + (uint64_t)((c * X_CHUNK_BYTES + kk * UMMA_K * 2) >> 4), idesc,
                                (pos != 0 || kk != 0) ? 1u : 0u);
            issued_any = true;
            if (++pos == spg || CPS * i + c == my_kt - 1) {
              tc_commit(acc_full(rr.slot));   // this group's sum is complete
              pos = 0;
              rr.advance(NACC);
            }
          }
        }
        if (!ok) break;
        tc_commit(a_empty(ra.slot));
        tc_commit(code_empty(rs.slot));
        ra.advance(ASTAGES);
        rs.advance(SSTAGES);
      }
      if (*abort_flag && issued_any) {
        tc_commit(drain_bar);
        if (!mbar_wait(drain_bar, 0, kDrainWaitNs, nullptr)) report_status(a.status, 5, kSiteW4Drain);
      }
    }
  } else {
    // ------------------------------------------------------------ dequantisation
    const int dg = (warp - 2) / 4;             // this warp's group: stages i = dg, dg + 2, ...
    const int quarter = warp % 4;
    const int n_local = quarter * 32 + lane;   // this thread's TMEM lane and W column
    const long long n = (long long)n0 + n_local;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    // bf16x2 -(128 + z): the sign bits set on the magic number plus the zero point
    const uint32_t negzz = (0x43004300u + (uint32_t)p.zero * 0x00010001u) ^ 0x80008000u;
    const unsigned short* sraw = reinterpret_cast<const unsigned short*>(p.scales);
    auto scale_raw = [&](int gl) -> uint32_t {
      return (gl < my_groups && n < a.N) ? (uint32_t)sraw[(long long)(g_begin + gl) * p.lds + n] : 0u;
    };
    // group 0 drains the accumulators in order, each scaled by its group's
    // scale (the raw bf16 bits of the next one are fetched a group ahead)
    int next_gl = 0;
    Ring rr;
    uint32_t s_cur = dg == 0 ? scale_raw(0) : 0u;
    auto consume_next = [&]() -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(rr.slot), rr.phase, a.timeout_ns, abort_flag))) {
        if (!*abort_flag) report_status(a.status, 5, kSiteW4Epilogue);
        *abort_flag = 1;
        return false;
      }
      tc_fence_after();
      uint32_t d[16];
      tmem_ld_32x32b_x16(lane_base + (uint32_t)(ACC_COL0 + rr.slot * MN), d);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(rr.slot));
      rr.advance(NACC);
      const float sc = __uint_as_float(s_cur << 16);
      s_cur = scale_raw(next_gl + 1);
#pragma unroll
      for (int m = 0; m < MN; ++m) acc[m] = fmaf(sc, __uint_as_float(d[m]), acc[m]);
      ++next_gl;
      return true;
    };
    bool ok = my_kt > 0;
    Ring rs, ra;
    for (int i = 0; i < dg; ++i) {   // this group's first stage
      rs.advance(SSTAGES);
      ra.advance(ASTAGES);
    }
    // wait results are made warp-uniform (__all_sync): a warp never splits
    // between leaving the loop and the warp-wide tcgen05/__syncwarp below
    for (int i = dg; ok && i < my_stages; i += DQ_GROUPS) {
      const bool got = mbar_wait(code_full(rs.slot), rs.phase, a.timeout_ns, abort_flag) &&
                       mbar_wait(a_empty(ra.slot), ra.phase ^ 1u, a.timeout_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (!*abort_flag) report_status(a.status, 5, kSiteW4Epilogue);
        *abort_flag = 1;
        ok = false;
        break;
      }
      const int nc = min(CPS, my_kt - CPS * i);
      const uint8_t* cp = base_ptr + (code_tile(rs.slot) - base) + n_local * (BK / 2);
      uint4 cw[CPS][2];
#pragma unroll
      for (int c = 0; c < CPS; ++c)
        if (c < nc) {
          cw[c][0] = *reinterpret_cast<const uint4*>(cp + c * CODE_CHUNK_BYTES);
          cw[c][1] = *reinterpret_cast<const uint4*>(cp + c * CODE_CHUNK_BYTES + 16);
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(code_empty(rs.slot));   // the codes are in registers
#pragma unroll
      for (int c = 0; c < CPS; ++c) {
        if (c < nc) {
          const uint32_t wds[8] = {cw[c][0].x, cw[c][0].y, cw[c][0].z, cw[c][0].w,
                                   cw[c][1].x, cw[c][1].y, cw[c][1].z, cw[c][1].w};
#pragma unroll
          for (int j2 = 0; j2 < 8; j2 += 2) {
            uint32_t t[8];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
              for (int h = 0; h < 4; ++h)
                t[jj * 4 + h] = fma1_bf16x2(and_or(wds[j2 + jj] >> (4 * h), 0x000F000Fu, 0x43004300u), negzz);
            tmem_st_x8(lane_base + (uint32_t)(ra.slot * A_COLS + c * (BK / 2) + j2 * 4), t);
          }
        }
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_full(ra.slot));
      // group 0: drain every group whose last chunk lies before this stage
      if (dg == 0) {
        while (ok && next_gl < my_groups && min((next_gl + 1) * spg, my_kt) <= CPS * i)
          ok = consume_next();
      }
      for (int k = 0; k < DQ_GROUPS; ++k) {
        rs.advance(SSTAGES);
        ra.advance(ASTAGES);
      }
    }
    if (dg == 0) {
      while (ok && next_gl < my_groups) ok = consume_next();
    }
  }

  // ---------------------------------------------------------------- reduction
  tc_fence_before();
  __syncthreads();  // every role has left the main loop: the ring may be reused
  if (threadIdx.x == 0) griddep_launch_dependents();
  const bool dq = warp >= 2 && warp < 6;   // the group holding the sums
  const int n_local = (warp % 4) * 32 + lane;
  if (p.split == 1) {
    if (dq && !*abort_flag) {
      const long long n = (long long)n0 + n_local;
      if (n < a.N) {
#pragma unroll
        for (int m = 0; m < MN; ++m)
          if (m < a.M) {
            float v = a.alpha * acc[m];
            if (a.beta != 0.f) v = fmaf(a.beta, load_out<OUT_BF16>(a, m, n), v);
            store_out<OUT_BF16>(a, m, n, v);
          }
      }
    }
  } else {
    if (dq) {
#pragma unroll
      for (int m = 0; m < MN; ++m) partial[m * BN + n_local] = acc[m];
    }
    cluster_sync();  // partials of every rank are visible cluster-wide
    // items of 4 columns of one row, over the columns this rank finishes
    const int cols = BN / p.split;
    const int groups4 = cols / 4;
    const int items = a.M * groups4;
    const uint32_t partial_addr = smem_u32(partial);
    for (int it = threadIdx.x; it < items; it += THREADS) {
      const int m = it / groups4;
      const int nl = rank * cols + (it % groups4) * 4;
      const uint32_t off = partial_addr + (uint32_t)(m * BN + nl) * 4u;
      float4 part[MAX_SPLIT];
#pragma unroll
      for (int q = 0; q < MAX_SPLIT; ++q)
        if (q < p.split) part[q] = ld_dsmem_f32x4(map_to_rank(off, (uint32_t)q));
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < MAX_SPLIT; ++q)
        if (q < p.split) {
          sum.x += part[q].x;
          sum.y += part[q].y;
          sum.z += part[q].z;
          sum.w += part[q].w;
        }
      const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
      const long long nn = (long long)n0 + nl;
      if (!*abort_flag) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (nn + e < a.N) {
            float v = a.alpha * sv[e];
            if (a.beta != 0.f) v = fmaf(a.beta, load_out<OUT_BF16>(a, m, nn + e), v);
            store_out<OUT_BF16>(a, m, nn + e, v);
          }
      }
    }
    cluster_sync();  // no rank leaves while others may still read its partial
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// --------------------------------------------------------------------- repack
// natural layout (codes packed along n, low nibble first) -> tiled layout,
// one 32-bit word per thread, padding tiles included (zero codes)
__global__ void __launch_bounds__(256) int4_repack_kernel(const uint8_t* __restrict__ q, long long ldq,
                                                          uint32_t* __restrict__ qk, int K, int N,
                                                          int k_tiles, long long words_total) {
  constexpr int kSlotK[8] = {0, 2, 4, 6, 1, 3, 5, 7};
  constexpr int WORDS_PER_ROW = BK / 8;                  // 8 words per column per tile
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < words_total;
       it += (long long)gridDim.x * blockDim.x) {
    // word it of the flat tiled array: tile, column inside it, word in the column
    const long long tile = it / (BN * WORDS_PER_ROW);
    const int r = (int)(it % (BN * WORDS_PER_ROW)) / WORDS_PER_ROW;
    const int j = (int)(it % WORDS_PER_ROW);
    const long long n = (tile / k_tiles) * BN + r;
    const int k0 = (int)(tile % k_tiles) * BK + 8 * j;
    uint32_t w = 0;
    if (n < N) {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int k = k0 + kSlotK[s];
        if (k < K) {
          const uint32_t b = q[(long long)k * ldq + n / 2];
          w |= ((b >> (4 * (n & 1))) & 0xFu) << (4 * s);
        }
      }
    }
    qk[it] = w;
  }
}

// --------------------------------------------------------------------- generic
// Any shape: one thread per C element, the same arithmetic (per-group fp32
// sums of x * (q - z), each scaled once).
template <bool OUT_BF16>
__global__ void __launch_bounds__(256) gemm_w4_generic_kernel(const W4Params p) {
  const GemmArgs& a = p.a;
  const long long total = (long long)a.M * a.N;
  const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(a.A);
  constexpr int kSlotOf[8] = {0, 4, 1, 5, 2, 6, 3, 7};   // nibble slot of k % 8
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const long long n = it % a.N;
    const int m = (int)(it / a.N);
    const uint8_t* col = p.qk + (size_t)(n / BN) * p.k_tiles * CODE_CHUNK_BYTES + (n % BN) * (BK / 2);
    float sum = 0.f;
    for (int g0 = 0; g0 < a.K; g0 += p.group) {
      const int g1 = min(g0 + p.group, a.K);
      float part = 0.f;
      for (int k = g0; k < g1; ++k) {
        const uint8_t* wp = col + (size_t)(k / BK) * CODE_CHUNK_BYTES + 4 * ((k % BK) / 8);
        const uint32_t w = (uint32_t)wp[0] | ((uint32_t)wp[1] << 8) | ((uint32_t)wp[2] << 16) |
                           ((uint32_t)wp[3] << 24);
        const int code = (int)((w >> (4 * kSlotOf[k % 8])) & 0xFu);
        part = fmaf(__bfloat162float(X[(long long)m * a.lda + k]), (float)(code - p.zero), part);
      }
      sum = fmaf(__bfloat162float(p.scales[(long long)(g0 / p.group) * p.lds + n]), part, sum);
    }
    float v = a.alpha * sum;
    if (a.beta != 0.f) v = fmaf(a.beta, load_out<OUT_BF16>(a, m, n), v);
    store_out<OUT_BF16>(a, m, n, v);
  }
}

int choose_split(int tiles_n, int groups, int num_sms) {
  // read once (a function-local static is initialised exactly once)
  static const int forced = [] {
    const char* e = std::getenv("GB300GEMM_W4_SPLIT");
    return e ? std::atoi(e) : 0;
  }();
  return plan::cluster_split(tiles_n, groups, num_sms, forced, MAX_SPLIT);
}

template <bool OUT_BF16>
int launch_fast(const W4Params& p0, const CUtensorMap* mapX, int num_sms, cudaStream_t s,
                int* k_split) {
  static std::atomic<uint64_t> smem_set{0};
  {
    cudaError_t e = set_smem_once(smem_set, gemm_w4_decode_kernel<OUT_BF16>, SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  W4Params p = p0;
  const int tiles_n = (p.a.N + BN - 1) / BN;
  if (tiles_n > 65535) return cudaErrorInvalidConfiguration;
  p.split = choose_split(tiles_n, p.groups, num_sms);
  *k_split = p.split;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.split, (unsigned)tiles_n, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_w4_decode_kernel<OUT_BF16>, *mapX, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool w4_fast_ok(int M, int K, int group) {
  return M >= 1 && M <= kSkMaxM && K >= 1 && (group % kW4BK == 0 || group >= K);
}

size_t w4_packed_bytes(int K, int N) {
  if (K <= 0 || N <= 0) return 0;
  return (size_t)((N + BN - 1) / BN) * ((K + BK - 1) / BK) * CODE_CHUNK_BYTES;
}

int launch_w4_decode(const GemmArgs& a, const void* scales, long long lds, int group, int zero,
                     const CUtensorMap* mapX, const uint8_t* qk, bool fast, int num_sms,
                     cudaStream_t s, int* k_split) {
  W4Params p;
  p.a = a;
  p.qk = qk;
  p.scales = static_cast<const __nv_bfloat16*>(scales);
  p.lds = lds;
  p.group = group;
  p.zero = zero;
  p.k_tiles = (a.K + BK - 1) / BK;
  p.stages_per_group = group >= a.K ? p.k_tiles : group / BK;
  p.groups = (a.K + group - 1) / group;
  p.split = 1;
  *k_split = 1;
  if (a.M <= 0 || a.N <= 0) return cudaSuccess;
  if (fast) {
    return a.out == Elem::BF16 ? launch_fast<true>(p, mapX, num_sms, s, k_split)
                               : launch_fast<false>(p, mapX, num_sms, s, k_split);
  }
  const long long total = (long long)a.M * a.N;
  const unsigned grid = (unsigned)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
  if (a.out == Elem::BF16)
    gemm_w4_generic_kernel<true><<<grid, 256, 0, s>>>(p);
  else
    gemm_w4_generic_kernel<false><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

int launch_int4_repack(const uint8_t* q, long long ldq, uint8_t* qk, int K, int N, int num_sms,
                       cudaStream_t s) {
  const long long total = (long long)(w4_packed_bytes(K, N) / 4);
  if (total <= 0) return cudaSuccess;
  const long long blocks = (total + 255) / 256;
  const unsigned grid = (unsigned)(blocks < (long long)num_sms * 8 ? blocks : (long long)num_sms * 8);
  int4_repack_kernel<<<grid, 256, 0, s>>>(q, ldq, reinterpret_cast<uint32_t*>(qk), K, N,
                                          (K + BK - 1) / BK, total);
  return cudaGetLastError();
}

}  // namespace g3
