// Interface between the C-ABI/dispatcher (gemm_api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace g3 {

// Raises `kernel`'s dynamic shared-memory limit to `bytes` once per device
// (the attribute belongs to the device's context); `done` holds one bit per
// device.  Two threads racing on the first call both set it, which is harmless.
template <class Kernel>
cudaError_t set_smem_once(std::atomic<uint64_t>& done, Kernel kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

enum class Elem : int { F32 = 0, BF16 = 1, FP8 = 2 };

// FP8 formats (values of gemm_fp8_format in the header).
enum Fp8Fmt : int { kE4M3 = 0, kE5M2 = 1 };

// Activations of the fused epilogue (values of gemm_activation in the header).
enum Act : int { kActNone = 0, kActRelu = 1, kActSilu = 2, kActGelu = 3 };

// One GEMM call after validation: C = alpha*A*B + beta*C, row-major.
struct GemmArgs {
  int M, N, K;
  float alpha, beta;
  const void* A;
  long long lda;
  const void* B;
  long long ldb;
  void* C;
  long long ldc;
  Elem in, out;
  int* status;          // device status word (one int, see report_status)
  uint64_t timeout_ns;  // bound on any single wait inside a kernel
  const float* bias;    // N fp32 values added to every row of C, or null
  int act;              // Act applied last
  const void* B2;       // SwiGLU: the up-projection (K x N, leading dimension ldb), else null
  int swiglu;           // 1: C = silu(A*B) * (A*B2) (alpha 1, beta 0, no bias)
  int fmt_a, fmt_b;     // in == FP8: the formats of A and B (Fp8Fmt)
  int stall;            // test hook: one role of the first CTA (or cluster) waits on a
                        // barrier nothing arrives at, so its bounded wait runs out and
                        // the kernel's abort path runs (tc2, skinny, FP32 SIMT kernels)
};

// Location codes recorded with a device timeout (bits 8 and up of the
// status word; the low 8 bits hold the gemm_status code).
enum WaitSite : int {
  kSiteSelftest = 1,
  kSiteTcProducer = 10,
  kSiteTcMma = 11,
  kSiteTcEpilogue = 12,
  kSiteTcDrain = 13,
  kSiteTc2Producer = 14,
  kSiteTc2Mma = 15,
  kSiteTc2Epilogue = 16,
  kSiteTc2Drain = 17,
  kSiteTc2StreamK = 18,    // a stream-K finisher pair waiting for another pair's partial tile
  kSiteSimtConsumer = 21,
  kSiteSimtDrain = 22,
  kSiteSimtStreamK = 23,   // a stream-K finisher waiting for another CTA's partial tile
  kSiteSkinnyProducer = 30,
  kSiteSkinnyMma = 31,
  kSiteSkinnyEpilogue = 32,
  kSiteSkinnyDrain = 33,
  kSiteW4Producer = 40,
  kSiteW4Mma = 41,
  kSiteW4Epilogue = 42,
  kSiteW4Drain = 43,
  kSiteAttnProducer = 50,
  kSiteAttnMma = 51,
  kSiteAttnSoftmax = 52,
  kSiteAttnDrain = 53,
};

// Each launcher returns a cudaError_t (as int) from the launch.
int launch_generic(const GemmArgs& a, cudaStream_t s);

// FP32 SIMT kernel: TMA tiles of A (16 k x 128 m, 64-byte swizzle) and
// B (bn n x 16 k), bn = 128 (8 x 8 register tiles, two CTAs per SM) or 256
// (8 x 16 register tiles, one CTA per SM).  plan_f32_simt picks the tile
// width (forced_tn 8 or 16 pins it, 0 lets the wave model choose) and
// whether the tiles of a partial last wave run as a second launch, K split
// over clusters of `split` CTAs (*k_split receives it; 1 otherwise).
struct SimtPlan {
  int tn = 8;     // register-tile width: 8 or 16 (C tiles of 128 x 16*tn)
  int split = 1;  // 1; 4 (narrow: clusters of four share a tile's K range);
                  // 0 (wide: stream-K over the SMs, partial tiles meeting in
                  // a per-device workspace)
};
// Lowers every stream-K flag of the current device's workspace (after a
// device timeout, which may leave flags raised).
void sk_clear_flags();
// The per-device stream-K workspace shared by the FP32 SIMT and CTA-pair
// kernels: stream_k_setup allocates and zeroes it at the first call on a
// device (a device-wide wait); stream_k_slot hands out its four slots in
// turn -- partial tiles (slot_floats floats, num_sms x 65536) and flags
// (slot_flags words, num_sms x 16, zero between calls).
cudaError_t stream_k_setup(int num_sms);
cudaError_t stream_k_slot(int num_sms, float** partials, unsigned** flags, size_t* slot_floats,
                          size_t* slot_flags);
int plan_f32_simt(int M, int N, int K, int num_sms, int forced_tn, SimtPlan* out);
int launch_f32_simt(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                    const SimtPlan& plan, int num_sms, cudaStream_t s, int* k_split);
constexpr int kSimtBM = 128, kSimtBK = 16, kSimtBN8 = 128, kSimtBN16 = 256;

// gemm_f32_noalloc: the FP32 SIMT plan run with the stream-K tail's partial
// tiles and flags in a static device array instead of the workspace, so the
// call allocates nothing.  The array holds the tail of up to
// kStaticScratchCtas CTAs; simt_stream_k_ctas gives the CTAs the tail of
// `plan` needs for this shape (0: the plan has no stream-K tail).
constexpr int kStaticScratchCtas = 152;
int simt_stream_k_ctas(int M, int N, int K, const SimtPlan& plan, int num_sms);
// Bytes of the static array (partial tiles and flags).
size_t simt_static_scratch_bytes();
// Plain GEMMs only (no bias or activation); the caller has checked that
// simt_stream_k_ctas() <= kStaticScratchCtas.
int launch_f32_simt_static(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                           const SimtPlan& plan, int num_sms, cudaStream_t s, int* k_split);

// BF16 tcgen05 kernel: TMA tiles of A (64 k x 128 m) and B (64 n x 64 k),
// 128-byte swizzle; C tiles of 128 x bn with bn from choose_tc_bn().
int choose_tc_bn(int M, int N, int num_sms);
// Single CTA (pair = 1) or CTA pair (pair = 2) and the tile width.
void choose_tc_config(int M, int N, int num_sms, int* pair, int* bn);
int launch_bf16_tc(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB, int bn,
                   int num_sms, cudaStream_t s);
constexpr int kTcBM = 128, kTcBK = 64;

// The same GEMM on CTA pairs (clusters of two, cta_group::2): C tiles of
// 256 x bn, bn in {128, 256}; each CTA loads 128 rows of A and bn/2 columns
// of B with the same tensor maps as the single-CTA kernel.
// *schedule receives 2 (whole tiles), 4 (the tiles of a partial last wave
// run as two half-width tiles each) or 6 (they run stream-K over the pairs).
bool split_tiles_enabled();
// gemm_force_split_tiles: 0 forbid, 1 automatic, 2 pin the CTA-pair
// kernel's stream-K tail, 3 pin its half-width tail (where each exists).
int split_tiles_mode();
int launch_bf16_tc_pair(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB, int bn,
                        int num_sms, cudaStream_t s, int* schedule);
// SwiGLU on CTA pairs (a.swiglu): C tiles of 256 x 128; each CTA's B operand
// is 64 columns of Bgate (mapB) and the same 64 columns of Bup (mapB2).
// FP8 inputs (in == FP8) on CTA pairs, 256 x 256 C tiles: TMA tiles of A
// (128 k x 128 m bytes) and B (128 n x 128 k bytes), 128-byte swizzle.
// *schedule as for launch_bf16_tc_pair (2 or 6: no half-width tiles).
int launch_fp8_tc_pair(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                       int num_sms, cudaStream_t s, int* schedule);
constexpr int kF8BK = 128;

int launch_bf16_swiglu_pair(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                            const CUtensorMap* mapB2, int num_sms, cudaStream_t s);

// Skinny (M <= 16) split-K kernel: TMA tiles of B (64 n x 64 k) and A
// (64 k x 16 rows), 128-byte swizzle.  mapB2 (the up-projection) is used
// when a.swiglu is set, and may be null otherwise.
// *k_split receives the number of CTAs K was split over.
int launch_skinny(const GemmArgs& a, const CUtensorMap* mapA, const CUtensorMap* mapB,
                  const CUtensorMap* mapB2, int num_sms, cudaStream_t s, int* k_split);
constexpr int kSkMaxM = 16, kSkBN = 128, kSkBK = 64;

// INT4 dequantisation W = s[k / G][n] * (q - z) (bf16 or fp32 W);
// *vector_path = 1 when the 32-codes-per-thread kernel ran.
int launch_int4_dequant(const uint8_t* q, int K, int N, int ldq, const void* scales, int lds,
                        int group, int zero, void* w, int ldw, bool out_bf16, int num_sms,
                        cudaStream_t st, int* vector_path);

// INT4 weight-only decode GEMM (bf16 X, M <= 16; codes in the tiled layout
// of 4 KB tiles, 128 columns x 64 rows of K): TMA tiles of X (64 k x 16 rows,
// 128-byte swizzle), bulk copies of the code tiles.  fast = the tcgen05
// kernel (w4_fast_ok and the alignment rules), else a one-thread-per-element
// kernel.
constexpr int kW4BN = 128, kW4BK = 64;
bool w4_fast_ok(int M, int K, int group);
size_t w4_packed_bytes(int K, int N);
int launch_w4_decode(const GemmArgs& a, const void* scales, long long lds, int group, int zero,
                     const CUtensorMap* mapX, const uint8_t* qk, bool fast, int num_sms,
                     cudaStream_t s, int* k_split);
// natural INT4 layout (packed along n) -> tiled layout (w4_packed_bytes)
int launch_int4_repack(const uint8_t* q, long long ldq, uint8_t* qk, int K, int N, int num_sms,
                       cudaStream_t s);

// Attention O = softmax(Q K^T * scale) V, [B][H][S][D] bf16 (K/V with Hkv
// heads).  fast = the tcgen05 kernel (D 64 or 128, 16-byte-aligned tensors;
// 3-D maps of Q with boxes 64 d x 128 rows and of K, V with 64 d x 64 keys),
// else a one-block-per-row kernel.
int launch_attention(int B, int Hq, int Hkv, int Sq, int Sk, int D, const void* Q, const void* K,
                     const void* V, void* O, float scale, int causal, const CUtensorMap* mQ,
                     const CUtensorMap* mK, const CUtensorMap* mV, bool fast, int* status,
                     uint64_t timeout_ns, cudaStream_t s);

int launch_selftest_wait(int* status, uint64_t timeout_ns, cudaStream_t s);

}  // namespace g3
