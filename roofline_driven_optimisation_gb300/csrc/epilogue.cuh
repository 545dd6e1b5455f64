// Elementwise epilogue shared by every kernel family: after the fp32
// accumulator acc of C[m][n] is final,
//
//     z = alpha*acc + beta*C_old[m][n] + bias[n]      (each term only if present)
//     C[m][n] = act(z)                                 (fp32, then one rounding)
//
// fused into the GEMM instead of a second pass over C ("Kernel 性能从何而来",
// section "优化 Memory-Bound Kernel": fuse the GEMM with its elementwise
// epilogue, so the intermediate never goes to HBM and back).
#pragma once
#include <cuda_runtime.h>

#include "internal.h"

namespace g3 {

__device__ __forceinline__ float activate(float z, int act) {
  switch (act) {
    case kActRelu:
      return fmaxf(z, 0.f);
    case kActSilu:  // z * sigmoid(z)
      return z / (1.f + expf(-z));
    case kActGelu:  // 0.5 z (1 + erf(z / sqrt 2))
      return 0.5f * z * (1.f + erff(z * 0.70710678118654752f));
    default:
      return z;
  }
}

// SwiGLU: silu(gate) * up
__device__ __forceinline__ float swiglu_combine(float gate, float up) {
  return gate / (1.f + expf(-gate)) * up;
}

// bias and activation of one value whose alpha/beta terms are already in v
__device__ __forceinline__ float finish(const GemmArgs& a, float v, long long n) {
  if (a.bias != nullptr) v += a.bias[n];
  return a.act == kActNone ? v : activate(v, a.act);
}

}  // namespace g3
