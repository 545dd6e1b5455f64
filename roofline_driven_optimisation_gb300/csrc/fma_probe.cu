// FP32 FMA throughput probe: the measured check on the FP32 roofline's
// compute peak.  "Kernel 性能从何而来" (section on the roofline model) bounds
// a compute-bound kernel by the hardware's peak arithmetic rate; for the
// CUDA-core path that peak is SMs x FP32 lanes x 2 FLOP x clock, and this
// kernel measures what the lanes actually retire, with the scalar FMA and
// with the packed fma.rn.f32x2 (two lanes per instruction), so the peak
// definition can be checked against both forms.
//
// Each thread runs CH independent two-lane FMA chains for `iters` rounds;
// nothing but the FMAs is in the loop.  The chains' values stay finite
// (multiplier within 1e-6 of 1) and a data-dependent store keeps the loop
// live.
#include <cuda_runtime.h>

#include <cstdint>

#include "gb300gemm_probe.h"

namespace {

constexpr int CH = 16;          // independent chains per thread (two lanes each)
constexpr int THREADS = 256;
constexpr int BLOCKS_PER_SM = 4;

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

template <bool PACKED>
__global__ void __launch_bounds__(THREADS) fma_rate_kernel(int iters, float* sink) {
  const float base = 1.0f + 1e-3f * (float)(threadIdx.x % 32);
  float sum = 0.f;
  if (PACKED) {
    uint64_t acc[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) acc[j] = pack2(base + j, base - 0.5f * j);
    const uint64_t mul = pack2(0.999999f, 1.000001f), add = pack2(1e-6f, -1e-6f);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int j = 0; j < CH; ++j) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[j]) : "l"(mul), "l"(add));
    }
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const float2 v = unpack2(acc[j]);
      sum += v.x + v.y;
    }
  } else {
    float lo[CH], hi[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      lo[j] = base + j;
      hi[j] = base - 0.5f * j;
    }
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        lo[j] = fmaf(lo[j], 0.999999f, 1e-6f);
        hi[j] = fmaf(hi[j], 1.000001f, -1e-6f);
      }
    }
#pragma unroll
    for (int j = 0; j < CH; ++j) sum += lo[j] + hi[j];
  }
  if (sum == 0.123456789f) sink[0] = sum;  // never true in practice; keeps the chains live
}

}  // namespace

extern "C" int gemm_probe_fp32_fma(int packed, int iters, float* sink, double* flops,
                                   cudaStream_t stream) {
  if (iters <= 0 || sink == nullptr || flops == nullptr) return 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 4;
  const unsigned blocks = (unsigned)sms * BLOCKS_PER_SM;
  if (packed)
    fma_rate_kernel<true><<<blocks, THREADS, 0, stream>>>(iters, sink);
  else
    fma_rate_kernel<false><<<blocks, THREADS, 0, stream>>>(iters, sink);
  if (cudaGetLastError() != cudaSuccess) return 4;
  *flops = (double)blocks * THREADS * (double)iters * CH * 2.0 /*lanes*/ * 2.0 /*FLOP per FMA*/;
  return 0;
}
