// Attention forward, O = softmax(Q K^T * scale) V, without materialising the
// score matrix.
//
// "从模型计算到 GPU 执行：读懂算子、Kernel 与 GPU 性能", section 1.2, writes
// attention as S = Q K^T, S = S / sqrt(d), P = softmax(S), O = P V.  "Kernel
// 性能从何而来", section on attention: the main cost of plain attention is
// writing S to HBM and reading it back; FlashAttention keeps the tiles on chip.
// Here a CTA owns 128 query rows of one head and walks the keys in tiles of
// 64, keeping S, P and O on chip and the softmax online (running row maximum
// m and sum l, O rescaled by exp(m_old - m_new) when the maximum moves):
//   * warp 0 streams Q once and the K/V tiles by TMA (two tiles ahead each),
//     warp 1 issues the tcgen05 MMAs, warps 2-5 are the softmax, one thread
//     per query row;
//   * S_j = Q K_j^T goes into one of two TMEM buffers (M = 128, N = 64), so
//     the MMA of tile j+1 runs while the softmax works on tile j;
//   * the softmax reads its row of S_j from TMEM, updates m and l in fp32,
//     writes P_j as bf16 back over the first half of the same TMEM buffer
//     (the P V MMA reads its A operand from tensor memory, so P never
//     passes through shared memory), and rescales its row of O in TMEM.  The reference
//     maximum m of a row moves only when a tile's maximum exceeds it by more
//     than TAU (log2 units): p = 2^(x - m) then stays below 2^TAU, O and l
//     share the reference, so O / l is unchanged, and the TMEM rescale of O
//     (a load, multiply and store of the whole row) becomes rare;
//   * O += P_j V_j accumulates in TMEM (M = 128, N = d); a warp whose rows
//     need no rescale releases P_j before the previous P V has finished, so
//     the P V MMAs run back to back; after the last tile each row is divided
//     by l and written as bf16;
//   * programmatic dependent launch: a CTA's set-up (barriers, tensor
//     memory) overlaps the previous kernel, and the next kernel's CTAs take
//     SM slots as this grid's CTAs leave.
// Masked scores (causal, or keys past Sk) are -inf before the softmax.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace g3 {
namespace {

constexpr int BM = 128;        // query rows per CTA
constexpr int BNK = 64;        // keys per tile
constexpr int KSTAGES = 2;     // K tiles in flight
constexpr int VSTAGES = 2;     // V tiles in flight
constexpr int THREADS = 192;   // producer, MMA, four softmax warps
constexpr int TMEM_COLS = 256; // two S buffers (2 x 64) + O (up to 128)
constexpr int S_COLS = BNK;
constexpr int O_COL0 = 2 * S_COLS;
constexpr float TAU = 8.f;     // lazy rescale threshold (p <= 2^TAU = 256)

template <int D>
struct AttnCfg {
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  static constexpr int BOXES = D / 64;                         // 64-column (128-byte) boxes of d
  static constexpr int Q_BYTES = BM * D * 2;                   // 16 / 32 KB
  static constexpr int KV_TILE_BYTES = BNK * D * 2;            // 8 / 16 KB
  static constexpr int SMEM_DATA = Q_BYTES + (KSTAGES + VSTAGES) * KV_TILE_BYTES;
  static constexpr int BAR_BYTES = 256;
  // padded so that at most two CTAs share an SM (their 2 x 256 tensor-memory
  // columns are then always free at allocation)
  static constexpr int SMEM_USED = SMEM_DATA + BAR_BYTES + 1024;
  static constexpr int SMEM_BYTES = SMEM_USED > 80 * 1024 ? SMEM_USED : 80 * 1024;
  static_assert(3 * (SMEM_BYTES + 1024) > 228 * 1024, "a third CTA must not fit");
};

struct AttnParams {
  int B, Hq, Hkv, Sq, Sk;
  float scale_log2;          // scale * log2(e)
  int causal;
  __nv_bfloat16* O;
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x by the special-function unit (ex2.approx, flush to zero): relative
// error about 2^-22, far below the bf16 rounding P takes next; 2^-inf = 0
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (two IEEE operations per instruction, round to
// nearest even, as the scalar forms).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                     const __grid_constant__ CUtensorMap mapV, const AttnParams p) {
  using Cfg = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t q_tile = base;
  auto k_tile = [&](int s) { return base + Cfg::Q_BYTES + s * Cfg::KV_TILE_BYTES; };
  auto v_tile = [&](int s) { return base + Cfg::Q_BYTES + (KSTAGES + s) * Cfg::KV_TILE_BYTES; };
  const uint32_t bar_base = base + Cfg::SMEM_DATA;
  uint8_t* bar_ptr = base_ptr + Cfg::SMEM_DATA;
  // barriers
  const uint32_t q_full = bar_base;
  auto k_full = [&](int s) { return bar_base + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar_base + 8u * (1 + KSTAGES + s); };
  constexpr int B0 = 1 + 2 * KSTAGES;
  auto v_full = [&](int s) { return bar_base + 8u * (B0 + s); };
  auto v_empty = [&](int s) { return bar_base + 8u * (B0 + VSTAGES + s); };
  constexpr int B1 = B0 + 2 * VSTAGES;
  auto s_full = [&](int b) { return bar_base + 8u * (B1 + b); };
  auto s_empty = [&](int b) { return bar_base + 8u * (B1 + 2 + b); };
  // P_j is released on p_full(j % 2).  Two barriers, not one: a warp that
  // needs no rescale releases P_j without waiting for P V of tile j - 1, so
  // it can reach tile j + 1 while another warp is still on tile j, and its
  // arrival must not count toward tile j's phase.  Tile j + 2 (the next
  // phase of the same barrier) needs S_{j+2}, which waits for P V of tile j.
  auto p_full = [&](int b) { return bar_base + 8u * (B1 + 4 + b); };
  // P V of tile j completes on o_done(j % 2): a warp waits every phase of
  // each, in order, and the next phase of the same barrier (tile j + 2)
  // cannot start before that warp has released P of tile j + 1, so a waiter
  // is never two phases behind
  auto o_done = [&](int b) { return bar_base + 8u * (B1 + 6 + b); };
  const uint32_t drain_bar = bar_base + 8u * (B1 + 8);
  constexpr int NBARS = B1 + 9;
  static_assert(NBARS * 8 + 16 <= AttnCfg<64>::BAR_BYTES, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_ptr + 8 * NBARS + 8);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // causal: the longest query tiles (last rows, most keys) of every head are
  // dispatched first and the short ones fill in behind them
  int qt = blockIdx.x, bh = blockIdx.y;             // query tile, b * Hq + h
  if (p.causal) {
    const int lin = blockIdx.y * gridDim.x + blockIdx.x;
    qt = gridDim.x - 1 - lin / gridDim.y;
    bh = lin % gridDim.y;
  }
  const int q0 = qt * BM;
  const int kvh = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / (p.Hq / p.Hkv);
  // keys this tile of queries can see: all, or (causal) up to its last row
  const int k_limit = p.causal ? min(p.Sk, q0 + BM + (p.Sk - p.Sq)) : p.Sk;
  const int n_tiles = k_limit > 0 ? (k_limit + BNK - 1) / BNK : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KSTAGES; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < VSTAGES; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_empty(b), 4);
      mbar_init(o_done(b), 1);
      mbar_init(p_full(b), 4);
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
  // launched with programmatic stream serialization: the set-up above
  // overlaps the end of the previous kernel on the stream; every read of Q,
  // K, V and every write of O comes after this wait.  The next kernel may be
  // scheduled as this grid's CTAs leave (it waits for this grid to finish
  // before touching memory).
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  auto fail_wait = [&](int site) {
    if (!*abort_flag) report_status(p.status, 5, site);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers
    // lane 0: Q and the K tiles, lane 1: the V tiles (two ahead each)
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      mbar_arrive_expect_tx(q_full, Cfg::Q_BYTES);
      for (int b = 0; b < Cfg::BOXES; ++b)
        tma_load_3d(q_tile + b * (BM * 128), &mapQ, q_full, b * 64, q0, bh);
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % KSTAGES;
        if (!mbar_wait(k_empty(s), (((uint32_t)(j / KSTAGES)) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
          fail_wait(kSiteAttnProducer);
          break;
        }
        mbar_arrive_expect_tx(k_full(s), Cfg::KV_TILE_BYTES);
        for (int b = 0; b < Cfg::BOXES; ++b)
          tma_load_3d(k_tile(s) + b * (BNK * 128), &mapK, k_full(s), b * 64, j * BNK, kvh);
      }
    } else if (lane == 1 && n_tiles > 0) {
      tma_prefetch_desc(&mapV);
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % VSTAGES;
        if (!mbar_wait(v_empty(s), (((uint32_t)(j / VSTAGES)) & 1u) ^ 1u, p.timeout_ns, abort_flag)) {
          fail_wait(kSiteAttnProducer);
          break;
        }
        mbar_arrive_expect_tx(v_full(s), Cfg::KV_TILE_BYTES);
        for (int b = 0; b < Cfg::BOXES; ++b)
          tma_load_3d(v_tile(s) + b * (BNK * 128), &mapV, v_full(s), b * 64, j * BNK, kvh);
      }
    }
    __syncwarp();
    // on an abort, copies in flight land on barriers nobody will wait for:
    // give them time before the shared memory is released
    if (lane == 0 && *abort_flag) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 50000) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_sync() && n_tiles > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BNK, 0, 0);   // Q K-major, K K-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, 0, 1);     // P in TMEM, V N-major
      bool ok = mbar_wait(q_full, 0, p.timeout_ns, abort_flag);
      bool issued_any = false;
      // S_j = Q K_j^T
      auto issue_s = [&](int j) -> bool {
        const int s = j % KSTAGES, b = j & 1;
        if (!mbar_wait(k_full(s), ((uint32_t)(j / KSTAGES)) & 1u, p.timeout_ns, abort_flag)) return false;
        if (j >= 2 && !mbar_wait(s_empty(b), (((uint32_t)(j / 2)) & 1u) ^ 1u, p.timeout_ns, abort_flag))
          return false;
        // S_j overwrites P_{j-2}, which P V of tile j-2 reads from tensor
        // memory; MMAs of different shapes are not ordered among themselves,
        // so that P V must have completed
        if (j >= 2 && !mbar_wait(o_done(b), (((uint32_t)(j / 2)) & 1u) ^ 1u, p.timeout_ns, abort_flag))
          return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t adesc = smem_desc_sw128(q_tile + (kk / 4) * (BM * 128) + (kk % 4) * 32, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(k_tile(s) + (kk / 4) * (BNK * 128) + (kk % 4) * 32, 16, 1024);
          tc_mma_f16(tmem_base + (uint32_t)(b * S_COLS), adesc, bdesc, idesc_s, kk != 0 ? 1u : 0u);
        }
        issued_any = true;
        tc_commit(k_empty(s));
        tc_commit(s_full(b));
        return true;
      };
      // O += P_j V_j
      auto issue_pv = [&](int j) -> bool {
        const int s = j % VSTAGES, b = j & 1;
        if (!mbar_wait(p_full(b), ((uint32_t)(j / 2)) & 1u, p.timeout_ns, abort_flag)) return false;
        if (!mbar_wait(v_full(s), ((uint32_t)(j / VSTAGES)) & 1u, p.timeout_ns, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BNK / 16; ++kk) {
          // A = P_j: TMEM lanes = rows, columns b*64 + kk*8 .. +7 = keys 16kk .. 16kk+15
          const uint32_t a_tmem = tmem_base + (uint32_t)(b * S_COLS + kk * 8);
          const uint64_t bdesc = smem_desc_sw128(v_tile(s) + kk * (16 * 128), BNK * 128, 1024);
          tc_mma_f16_tmem_a(tmem_base + (uint32_t)O_COL0, a_tmem, bdesc, idesc_o, (j | kk) != 0 ? 1u : 0u);
        }
        issued_any = true;
        tc_commit(v_empty(s));
        tc_commit(o_done(b));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 1; ok && j < n_tiles; ++j) {
        ok = issue_s(j);
        if (ok) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(n_tiles - 1);
      if (!ok) {
        fail_wait(kSiteAttnMma);
        if (issued_any) {
          tc_commit(drain_bar);
          if (!mbar_wait(drain_bar, 0, kDrainWaitNs, nullptr)) report_status(p.status, 5, kSiteAttnDrain);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax, one thread per row
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;            // row inside the tile = TMEM lane
    const int qi = q0 + r;                        // query index
    const int vis_last = p.causal ? qi + (p.Sk - p.Sq) : p.Sk - 1;   // last visible key
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // every wait result is made warp-uniform (__all_sync), so a warp never
    // splits between leaving the loop and the warp-wide operations below
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int b = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full(b), ((uint32_t)(j / 2)) & 1u, p.timeout_ns, abort_flag))) {
        fail_wait(kSiteAttnSoftmax);
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sa[32], sb[32];
      tmem_ld_32x32b_x32(lane_base + (uint32_t)(b * S_COLS), sa);
      tmem_ld_32x32b_x32(lane_base + (uint32_t)(b * S_COLS + 32), sb);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty(b));
      // raw scores, masked (-inf) only on tiles that need it; the scale is
      // applied inside the exponent's FMA below
      float sv[64];
      const int k0 = j * BNK;
      if (k0 + BNK - 1 <= min(vis_last, p.Sk - 1)) {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = __uint_as_float(c < 32 ? sa[c] : sb[c - 32]);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int kj = k0 + c;
          const bool vis = kj < p.Sk && kj <= vis_last;
          sv[c] = vis ? __uint_as_float(c < 32 ? sa[c] : sb[c - 32]) : -INFINITY;
        }
      }
      // row maximum of the raw scores over eight independent partials (the
      // scale is positive, so the maximum of the scaled scores is this one
      // scaled, exactly: rounding is monotonic)
      float red[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        red[i] = fmax3(sv[i], sv[8 + i], sv[16 + i]);
        red[i] = fmax3(red[i], sv[24 + i], sv[32 + i]);
        red[i] = fmax3(red[i], sv[40 + i], sv[48 + i]);
        red[i] = fmaxf(red[i], sv[56 + i]);
      }
      const float mt = fmax3(fmax3(red[0], red[1], red[2]), fmax3(red[3], red[4], red[5]),
                             fmaxf(red[6], red[7])) * p.scale_log2;
      // move the reference maximum only when this tile exceeds it by > TAU
      const bool move = mt > m + TAU;       // also the first visible tile (m = -inf)
      const float m_new = move ? mt : m;
      const float m_use = m_new == -INFINITY ? 0.f : m_new;   // no visible key yet
      const float alpha = move ? ex2_approx(m - m_use) : 1.f;  // 0 on the first visible tile
      // p = 2^(s * scale - m): the argument of two keys in one packed FMA,
      // the row sum over four packed (eight scalar) partials
      const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
      const uint64_t negm2 = f2_pack(-m_use, -m_use);
      uint64_t sum2[4];
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 arg = f2_unpack(ffma2(f2_pack(sv[c], sv[c + 1]), scale2, negm2));
        const float p0 = ex2_approx(arg.x), p1 = ex2_approx(arg.y);
        const uint64_t pp = f2_pack(p0, p1);
        sum2[(c / 2) % 4] = c < 8 ? pp : fadd2(sum2[(c / 2) % 4], pp);
        pw[c / 2] = pack_bf16x2(p0, p1);
      }
      const float2 s01 = f2_unpack(fadd2(sum2[0], sum2[1])), s23 = f2_unpack(fadd2(sum2[2], sum2[3]));
      const float psum = (s01.x + s01.y) + (s23.x + s23.y);
      l = l * alpha + psum;
      m = m_new;
      // P_j over the first 32 columns of its S buffer (two keys per column)
      tmem_st_32x32b_x32(lane_base + (uint32_t)(b * S_COLS), pw);
      tc_wait_st();
      // O is touched only to rescale it; the warp decides together
      const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
      if (!rescale) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(b));
      }
      // every P V phase is observed in order (see o_done)
      if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(o_done((j - 1) & 1), ((uint32_t)((j - 1) / 2)) & 1u,
                                                      p.timeout_ns, abort_flag))) {
        fail_wait(kSiteAttnSoftmax);
        ok = false;
        break;
      }
      if (rescale) {
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(lane_base + (uint32_t)(O_COL0 + c0), o);
          tc_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_32x32b_x32(lane_base + (uint32_t)(O_COL0 + c0), o);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(b));
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n_tiles > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(o_done((n_tiles - 1) & 1), ((uint32_t)((n_tiles - 1) / 2)) & 1u,
                                             p.timeout_ns, abort_flag))) {
        fail_wait(kSiteAttnSoftmax);
        ok = false;
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    // every lane of the warp loads (tcgen05.ld is warp-wide); only rows
    // inside the sequence store, and nothing is stored after a timeout
    const bool write = __all_sync(0xffffffffu, ok && !*abort_flag);
    if (write) {
      __nv_bfloat16* orow = p.O + ((size_t)bh * p.Sq + qi) * D;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        if (n_tiles > 0) {
          tmem_ld_32x32b_x32(lane_base + (uint32_t)(O_COL0 + c0), o);
          tc_wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0u;
        }
        if (qi >= p.Sq) continue;
        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                              pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                              pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                              pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
      }
    }
    // after a device timeout nothing is written
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ generic
// Any head dimension or alignment: one block per (head, query row); the row's
// scores live in shared memory (Sk floats), then max, sum and P V.
__global__ void __launch_bounds__(128) attention_generic_kernel(const __nv_bfloat16* __restrict__ Q,
                                                                const __nv_bfloat16* __restrict__ K,
                                                                const __nv_bfloat16* __restrict__ V,
                                                                __nv_bfloat16* __restrict__ O, int Hq,
                                                                int Hkv, int Sq, int Sk, int D, float scale,
                                                                int causal) {
  extern __shared__ float sc[];   // Sk scores, then 32 floats of reduction space
  float* red = sc + Sk;
  const int qi = blockIdx.x, bh = blockIdx.y;
  const int kvh = (bh / Hq) * Hkv + (bh % Hq) / (Hq / Hkv);
  const __nv_bfloat16* q = Q + ((size_t)bh * Sq + qi) * D;
  const __nv_bfloat16* kb = K + (size_t)kvh * Sk * D;
  const __nv_bfloat16* vb = V + (size_t)kvh * Sk * D;
  const int vis_last = causal ? qi + (Sk - Sq) : Sk - 1;
  const int nvis = min(Sk, vis_last + 1);
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < Sk; j += blockDim.x) {
    float s = -INFINITY;
    if (j < nvis) {
      float acc = 0.f;
      for (int t = 0; t < D; ++t) acc = fmaf(__bfloat162float(q[t]), __bfloat162float(kb[(size_t)j * D + t]), acc);
      s = acc * scale;
    }
    sc[j] = s;
    mx = fmaxf(mx, s);
  }
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float sum = 0.f;
  for (int j = threadIdx.x; j < Sk; j += blockDim.x) {
    const float e = j < nvis ? expf(sc[j] - mx) : 0.f;
    sc[j] = e;
    sum += e;
  }
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = sum;
  __syncthreads();
  sum = red[0] + red[1] + red[2] + red[3];
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __nv_bfloat16* orow = O + ((size_t)bh * Sq + qi) * D;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < nvis; ++j) acc = fmaf(sc[j], __bfloat162float(vb[(size_t)j * D + c]), acc);
    orow[c] = __float2bfloat16_rn(acc * inv);
  }
}

template <int D>
int launch_fast(const AttnParams& p, const CUtensorMap* mQ, const CUtensorMap* mK, const CUtensorMap* mV,
                cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_smem_once(smem_set, attention_kernel<D>, AttnCfg<D>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)((p.Sq + BM - 1) / BM), (unsigned)(p.B * p.Hq));
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = AttnCfg<D>::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attention_kernel<D>, *mQ, *mK, *mV, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int launch_attention(int B, int Hq, int Hkv, int Sq, int Sk, int D, const void* Q, const void* K,
                     const void* V, void* O, float scale, int causal, const CUtensorMap* mQ,
                     const CUtensorMap* mK, const CUtensorMap* mV, bool fast, int* status,
                     uint64_t timeout_ns, cudaStream_t s) {
  if (B == 0 || Hq == 0 || Sq == 0) return cudaSuccess;
  if (fast) {
    AttnParams p;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Sk = Sk;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal;
    p.O = static_cast<__nv_bfloat16*>(O);
    p.status = status;
    p.timeout_ns = timeout_ns;
    return D == 128 ? launch_fast<128>(p, mQ, mK, mV, s) : launch_fast<64>(p, mQ, mK, mV, s);
  }
  const size_t smem = ((size_t)Sk + 32) * sizeof(float);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(attention_generic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)Sq, (unsigned)(B * Hq));
  attention_generic_kernel<<<grid, 128, smem, s>>>(
      static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
      static_cast<const __nv_bfloat16*>(V), static_cast<__nv_bfloat16*>(O), Hq, Hkv, Sq, Sk, D, scale, causal);
  return cudaGetLastError();
}

}  // namespace g3
