// Decode-shaped GEMM (M <= 16 rows of activations against a K x N weight):
// C = alpha*A*B + beta*C with bf16 A (M x K), bf16 B (K x N), fp32
// accumulation, bf16 or fp32 C.
//
// With M this small the arithmetic intensity is about M FLOP per byte of B,
// far left of the ridge point, so the kernel is judged by HBM bandwidth
// ("CUDA 算子工程 ch.4 内存层级与代价表", 4.6: small-batch GEMM is
// bandwidth-bound; "Kernel 性能从何而来", section "优化 Memory-Bound Kernel":
// move every byte once, use TMA for regular tiles, keep enough requests in
// flight).  Design:
//   * each B element is read from HBM exactly once, by TMA, into a 6-stage
//     shared-memory ring (16 KB of B per stage), with an evict-first L2 hint;
//   * the math runs on the tensor cores with the operands swapped,
//     D^T = B^T A^T: the 128-column slab of B is the MMA's M = 128 operand
//     (N-major in shared memory) and the <= 16 activation rows are the
//     MMA's N = 16 operand (K-major), so no shuffle of B is needed and the
//     tensor pipe has far more throughput than the stream needs;
//   * K is split over the CTAs of a thread-block cluster (split S <= 8);
//     each CTA leaves its 128 x 16 fp32 partial in its own shared memory and
//     the partials are summed across the cluster through distributed shared
//     memory in rank order 0..S-1 -- a fixed order, so results are
//     bit-reproducible, and no global workspace is used;
//   * the beta*C residual and the conversion are fused into that reduction
//     (same page, section "优化 Memory-Bound Kernel": fuse the elementwise
//     epilogue instead of a second pass over C); the two warps that have no
//     role in the main loop fetch their C values into registers while the
//     weights stream, so that read is off the kernel's tail;
//   * launched with programmatic stream serialization: the launch, barrier
//     set-up, TMEM allocation and an L2 prefetch of the first weight stages
//     overlap the previous kernel on the stream, and every read into the SM
//     waits on griddepcontrol.wait.
// SwiGLU variant (SW): C = silu(A*Bgate) * (A*Bup) for 64 output columns per
// CTA.  The MMA's 128 rows are those 64 columns of Bgate followed by the
// same 64 columns of Bup (one TMA box from each weight), so the stage size,
// the MMA and the TMEM layout are unchanged; the two halves of the
// accumulator meet in the reduction, which applies silu(g) * u before the
// single rounding to bf16.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>

#include "epilogue.cuh"
#include "internal.h"
#include "plan.h"
#include "ptx.cuh"

namespace g3 {
namespace {

constexpr int BN = kSkBN;    // B columns per CTA (MMA M)
constexpr int BK = kSkBK;    // K per stage
constexpr int MN = kSkMaxM;  // MMA N: activation rows, zero-padded by TMA
#ifndef GB300_SKINNY_STAGES
#define GB300_SKINNY_STAGES 6
#endif
constexpr int STAGES = GB300_SKINNY_STAGES;
constexpr int UMMA_K = 16;
constexpr int B_BOX_BYTES = 64 * BK * 2;                 // 8 KB: 64 columns x 64 k
constexpr int B_STAGE_BYTES = BN * BK * 2;               // 16 KB
constexpr int A_STAGE_BYTES = MN * BK * 2;               // 2 KB
constexpr int STAGE_BYTES = B_STAGE_BYTES + A_STAGE_BYTES;
constexpr int THREADS = 128;
constexpr int TMEM_COLS = 32;
constexpr int PARTIAL_BYTES = MN * BN * 4;               // 8 KB, aliases stage 0 after the main loop
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 256 + 1024;
constexpr int MAX_SPLIT = 8;
// split > 1: a reduction item is 4 adjacent columns of one row; 128 threads
// cover the 16 x 128 tile with at most RED_ITEMS items each
constexpr int RED_ITEMS = MN * BN / 4 / THREADS;
static_assert(PARTIAL_BYTES <= STAGE_BYTES, "partial tile aliases one stage");
static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned");

// The raw bits of C_old (bf16 zero-extended, or fp32): the load writes the
// register directly, so nothing waits for it until raw_to_float() runs.
template <bool OUT_BF16>
__device__ __forceinline__ uint32_t load_c_raw(const GemmArgs& a, int m, long long n) {
  const long long off = (long long)m * a.ldc + n;
  if (OUT_BF16) return static_cast<const unsigned short*>(a.C)[off];
  return __float_as_uint(static_cast<const float*>(a.C)[off]);
}
template <bool OUT_BF16>
__device__ __forceinline__ float raw_to_float(uint32_t w) {
  return OUT_BF16 ? __uint_as_float(w << 16) : __uint_as_float(w);
}

// SwiGLU output: silu(gate) * up rounded once to bf16
__device__ __forceinline__ void store_swiglu(const GemmArgs& a, int m, long long n, float gate, float up) {
  static_cast<__nv_bfloat16*>(a.C)[(long long)m * a.ldc + n] = __float2bfloat16_rn(swiglu_combine(gate, up));
}

template <bool OUT_BF16>
__device__ __forceinline__ void store_c(const GemmArgs& a, int m, long long n, float v) {
  v = finish(a, v, n);
  const long long off = (long long)m * a.ldc + n;
  if (OUT_BF16)
    static_cast<__nv_bfloat16*>(a.C)[off] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(a.C)[off] = v;
}

struct SkinnyParams {
  GemmArgs a;
  int split;       // CTAs per cluster along K
  int k_tiles;     // total K stages
  int c_vec;       // unused by the scalar stores; kept for symmetry
};

// Sum over the S ranks of the cluster, in rank order, of the 16-byte piece
// at shared address `off` of each rank's partial tile; all S loads are in
// flight before the first add.
__device__ __forceinline__ float4 sum_ranks(uint32_t off, int split) {
  float4 part[MAX_SPLIT];
#pragma unroll
  for (int q = 0; q < MAX_SPLIT; ++q)
    if (q < split) part[q] = ld_dsmem_f32x4(map_to_rank(off, (uint32_t)q));
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < MAX_SPLIT; ++q)
    if (q < split) {
      sum.x += part[q].x;
      sum.y += part[q].y;
      sum.z += part[q].z;
      sum.w += part[q].w;
    }
  return sum;
}

// mapB2 is read only by the SwiGLU variant (the up-projection).
template <bool OUT_BF16, bool SW>
__global__ void __launch_bounds__(THREADS, 2)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap mapA,
                       const __grid_constant__ CUtensorMap mapB,
                       const __grid_constant__ CUtensorMap mapB2, const SkinnyParams p) {
  static_assert(!SW || OUT_BF16, "the SwiGLU variant writes bf16");
  constexpr int OUT_COLS = SW ? BN / 2 : BN;  // C columns per CTA
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bar_base = base + STAGES * STAGE_BYTES;
  uint8_t* bar_ptr = base_ptr + STAGES * STAGE_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  const uint32_t tfull_bar = bar_base + 8u * (2 * STAGES);
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * STAGES + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_ptr + 8 * (2 * STAGES + 2) + 8);
  const uint32_t stall_bar = bar_base + 8u * (2 * STAGES + 4);  // test hook: nothing arrives
  static_assert(8 * (2 * STAGES + 5) <= 256, "barrier area");
  auto b_tile = [&](int s) { return base + s * STAGE_BYTES; };
  auto a_tile = [&](int s) { return base + s * STAGE_BYTES + B_STAGE_BYTES; };
  float* partial = reinterpret_cast<float*>(base_ptr);  // [MN][BN], valid after the main loop

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const GemmArgs& a = p.a;
  const int rank = (int)cluster_ctarank();          // position along K inside the cluster
  const int n0 = blockIdx.y * OUT_COLS;
  // TMA box j of a stage: 64 columns of B (or, SwiGLU, of Bgate then Bup)
  auto box_map = [&](int j) { return (SW && j == 1) ? &mapB2 : &mapB; };
  auto box_col = [&](int j) { return SW ? n0 : n0 + j * 64; };
  const int kt_begin = (int)((long long)p.k_tiles * rank / p.split);
  const int kt_end = (int)((long long)p.k_tiles * (rank + 1) / p.split);
  const int my_kt = kt_end - kt_begin;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    mbar_init(stall_bar, 1);
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
    // While the previous kernel on the stream finishes, pull the first
    // stages of this CTA's weights into L2 (a prefetch only: the real loads
    // come after the wait and see whatever is in memory then).
    tma_prefetch_desc(&mapB);
    if (SW) tma_prefetch_desc(&mapB2);
    const int pre = my_kt < STAGES ? my_kt : STAGES;
    for (int kt = kt_begin; kt < kt_begin + pre; ++kt)
#pragma unroll
      for (int j = 0; j < BN / 64; ++j) tma_prefetch_l2_2d(box_map(j), box_col(j), kt * BK);
  }
  griddep_wait();  // inputs may come from the previous kernel on the stream

  // C_old of this thread's outputs, loaded now and not used until the
  // epilogue, so the loads stay in flight while the weights stream (no
  // thread -- in particular not the TMA producer -- waits for them here).
  // split == 1: column n0 + threadIdx.x, rows 0..M-1.  split > 1: items of 4
  // columns of the columns this rank finishes.
  const int cols = OUT_COLS / p.split;
  const int groups = cols / 4;
  const int items = a.M * groups;
  uint32_t cpre[MN];  // split == 1: one per row; split > 1: RED_ITEMS x 4
  static_assert(RED_ITEMS * 4 <= MN, "prefetch registers");
#pragma unroll
  for (int j = 0; j < MN; ++j) cpre[j] = 0u;
  if (!SW && a.beta != 0.f) {
    if (p.split == 1) {
      const long long n = (long long)n0 + threadIdx.x;
#pragma unroll
      for (int m = 0; m < MN; ++m)
        if (m < a.M && n < a.N) cpre[m] = load_c_raw<OUT_BF16>(a, m, n);
    } else {
#pragma unroll
      for (int j = 0; j < RED_ITEMS; ++j) {
        const int it = threadIdx.x + j * THREADS;
        if (it < items) {
          const int m = it / groups;
          const long long n = (long long)n0 + rank * cols + (it % groups) * 4;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n + e < a.N) cpre[j * 4 + e] = load_c_raw<OUT_BF16>(a, m, n + e);
        }
      }
    }
  }

  if (warp == 0) {
    if (elect_one_sync() && my_kt > 0) {
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapB);
      if (SW) tma_prefetch_desc(&mapB2);
      const uint64_t stream_policy = l2_policy_evict_first();
      // bit s of `issued`: slot s has had a copy issued; bit s of
      // `issued_par`: the phase parity of its latest copy
      uint32_t issued = 0, issued_par = 0;
      int stage = 0;
      uint32_t phase = 0;
      for (int kt = kt_begin; kt < kt_end; ++kt) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, a.timeout_ns, abort_flag)) {
          if (!*abort_flag) report_status(a.status, 5, kSiteSkinnyProducer);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
#pragma unroll
        for (int j = 0; j < BN / 64; ++j)
          tma_load_2d_hint(b_tile(stage) + j * B_BOX_BYTES, box_map(j), full_bar(stage), box_col(j),
                           kt * BK, stream_policy);
        tma_load_2d(a_tile(stage), &mapA, full_bar(stage), kt * BK, 0);
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < STAGES; ++s)
          if (((issued >> s) & 1u) &&
              !mbar_wait(full_bar(s), (issued_par >> s) & 1u, kDrainWaitNs, nullptr))
            report_status(a.status, 5, kSiteSkinnyDrain);
      }
    }
  } else if (warp == 1) {
    if (elect_one_sync() && my_kt > 0) {
      // D^T (128 x 16) += B^T (128 x 16, N-major) * A^T (16 x 16, K-major)
      constexpr uint32_t idesc = idesc_bf16_f32(BN, MN, /*A MN-major*/ 1, /*B K-major*/ 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      if (a.stall && rank == 0 && blockIdx.y == 0 &&
          !mbar_wait(stall_bar, 0, a.timeout_ns / 4, abort_flag)) {
        // test hook: this wait runs out; the cluster takes its abort path
        if (!*abort_flag) report_status(a.status, 5, kSiteSkinnyMma);
        *abort_flag = 1;
        ok = false;
      }
      for (int kt = 0; ok && kt < my_kt; ++kt) {
        if (!mbar_wait(full_bar(stage), phase, a.timeout_ns, abort_flag)) {
          if (!*abort_flag) report_status(a.status, 5, kSiteSkinnyMma);
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(b_tile(stage) + kk * UMMA_K * 128, B_BOX_BYTES, 1024);
          const uint64_t adesc = smem_desc_sw128(a_tile(stage) + kk * UMMA_K * 2, 16, 1024);
          tc_mma_f16(tmem_base, bdesc, adesc, idesc, (kt | kk) != 0 ? 1u : 0u);
        }
        tc_commit(empty_bar(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        tc_commit(tfull_bar);
      } else {
        tc_commit(drain_bar);
        if (!mbar_wait(drain_bar, 0, kDrainWaitNs, nullptr)) report_status(a.status, 5, kSiteSkinnyDrain);
      }
    }
  }

  // ---------------------------------------------------------------- partials
  // All four warps: TMEM lanes [32w, 32w+32) hold columns n0+32w+lane of
  // D^T, one fp32 per activation row.
  __syncwarp();
  bool have = false;
  if (my_kt > 0) {
    have = mbar_wait(tfull_bar, 0, a.timeout_ns, abort_flag);
    if (!have && !*abort_flag) {
      report_status(a.status, 5, kSiteSkinnyEpilogue);
      *abort_flag = 1;
    }
  }
  __syncwarp();
  tc_fence_after();
  __syncthreads();  // every role has left the main loop: stage 0 may now be reused
  uint32_t r[16];
  if (my_kt > 0 && !*abort_flag) {
    tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(warp * 32) << 16), r);
    tc_wait_ld();
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) r[j] = 0u;
  }
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (!SW && p.split == 1) {
    // the whole K range is in this CTA: column n0 + threadIdx.x of C is in
    // this thread's registers, one value per activation row
    const long long n = (long long)n0 + threadIdx.x;
    if (n < a.N) {
#pragma unroll
      for (int m = 0; m < MN; ++m)
        if (m < a.M)
          store_c<OUT_BF16>(a, m, n,
                            fmaf(a.alpha, __uint_as_float(r[m]), a.beta * raw_to_float<OUT_BF16>(cpre[m])));
    }
  } else {
    const int n_local = warp * 32 + lane;
#pragma unroll
    for (int m = 0; m < MN; ++m) partial[m * BN + n_local] = __uint_as_float(r[m]);
    cluster_sync();  // partials of every rank are visible cluster-wide
    const uint32_t partial_addr = smem_u32(partial);
    // the sums first (every read of another rank's shared memory), then this
    // rank says it is done reading, then the stores: the stores overlap the
    // wait for the other ranks, and no rank leaves while others may still
    // read its partial
    float4 sum[RED_ITEMS], up[SW ? RED_ITEMS : 1];
#pragma unroll
    for (int j = 0; j < RED_ITEMS; ++j) {
      const int it = threadIdx.x + j * THREADS;
      if (it < items) {
        const int m = it / groups;
        const int nl = rank * cols + (it % groups) * 4;
        const uint32_t off = partial_addr + (uint32_t)(m * BN + nl) * 4u;
        sum[j] = sum_ranks(off, p.split);
        // SwiGLU: the up-projection of the same columns is 64 rows further down D^T
        if (SW) up[SW ? j : 0] = sum_ranks(off + (uint32_t)(BN / 2) * 4u, p.split);
      }
    }
    cluster_arrive();
#pragma unroll
    for (int j = 0; j < RED_ITEMS; ++j) {
      const int it = threadIdx.x + j * THREADS;
      if (it < items) {
        const int m = it / groups;
        const int nl = rank * cols + (it % groups) * 4;
        const long long n = (long long)n0 + nl;
        const float sv[4] = {sum[j].x, sum[j].y, sum[j].z, sum[j].w};
        if (SW) {
          const float4 u = up[SW ? j : 0];
          const float uv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n + e < a.N) store_swiglu(a, m, n + e, sv[e], uv[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (n + e < a.N)
              store_c<OUT_BF16>(a, m, n + e,
                                fmaf(a.alpha, sv[e], a.beta * raw_to_float<OUT_BF16>(cpre[j * 4 + e])));
        }
      }
    }
    cluster_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

int choose_split(int tiles_n, int k_tiles, int num_sms) {
  // read once (a function-local static is initialised exactly once)
  static const int forced = [] {
    const char* e = std::getenv("GB300GEMM_SKINNY_SPLIT");
    return e ? std::atoi(e) : 0;
  }();
  return plan::cluster_split(tiles_n, k_tiles, num_sms, forced, MAX_SPLIT);
}

template <bool OUT_BF16, bool SW>
int launch_impl(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                const CUtensorMap* mapB2, int num_sms, cudaStream_t s, int* k_split) {
  constexpr int OUT_COLS = SW ? BN / 2 : BN;
  static std::atomic<uint64_t> smem_set{0};
  {
    cudaError_t e = set_smem_once(smem_set, gemm_skinny_kernel<OUT_BF16, SW>, SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  SkinnyParams p;
  p.a = a;
  p.k_tiles = (a.K + BK - 1) / BK;
  const int tiles_n = (a.N + OUT_COLS - 1) / OUT_COLS;
  if (tiles_n <= 0 || a.M <= 0) return cudaSuccess;
  if (tiles_n > 65535) return cudaErrorInvalidConfiguration;
  p.split = choose_split(tiles_n, p.k_tiles, num_sms);
  *k_split = p.split;
  p.c_vec = 0;

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
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<OUT_BF16, SW>, *mapA, *mapB,
                                     SW ? *mapB2 : *mapB, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int launch_skinny(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                  const CUtensorMap* mapB2, int num_sms, cudaStream_t s, int* k_split) {
  *k_split = 1;
  if (a.swiglu) {
    if (a.out != Elem::BF16 || mapB2 == nullptr) return cudaErrorInvalidValue;
    return launch_impl<true, true>(a, mapA, mapB, mapB2, num_sms, s, k_split);
  }
  if (a.out == Elem::BF16) return launch_impl<true, false>(a, mapA, mapB, nullptr, num_sms, s, k_split);
  return launch_impl<false, false>(a, mapA, mapB, nullptr, num_sms, s, k_split);
}

}  // namespace g3
