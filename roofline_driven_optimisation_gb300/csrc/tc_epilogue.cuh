// Parameters and epilogue shared by the two tensor-core GEMM kernels
// (single-CTA and CTA-pair): one thread owns one row of the C tile and turns
// 32 fp32 accumulator columns into C = alpha*acc + beta*C_old, evaluated in
// fp32 and rounded once to the output type, written with 16-byte stores when
// the row segment is aligned and complete ("Kernel 性能从何而来", section
// "优化 Memory-Bound Kernel": the elementwise epilogue is fused into the GEMM).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "epilogue.cuh"
#include "internal.h"

namespace g3 {
namespace {

struct TcParams {
  GemmArgs a;
  int tiles_m, tiles_n, num_tiles, k_tiles;
  int c_vec;       // C 16-byte aligned and ldc*sizeof(out) a multiple of 16
  // CTA-pair kernel: tiles [0, dp_tiles) run one per pair; the remaining
  // tiles run as half_tiles items of half the width, one per pair
  int dp_tiles;
  int half_tiles;
  // or (stream-K instance) the K-steps of tiles [dp_tiles, num_tiles) run
  // end to end over sk_pairs pairs, partial tiles meeting in a workspace slot
  int sk_pairs = 0;
  long long sk_units = 0;
  float* sk_partials = nullptr;   // [pair][2 pieces][256 rows][BN] fp32
  unsigned* sk_flags = nullptr;   // [pair][2 pieces][2 CTAs x 4 epilogue warps]
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Epilogue for one row segment of 32 columns: v = alpha*acc (+ beta*C_old).
template <bool OUT_BF16>
__device__ __forceinline__ void store_row32(const TcParams& p, long long m, long long n,
                                            const uint32_t (&r)[32]) {
  const GemmArgs& a = p.a;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = a.alpha * __uint_as_float(r[j]);
  const bool beta_nz = a.beta != 0.f;
  const bool full = p.c_vec && (n + 32 <= a.N);
  const bool epi = a.bias != nullptr || a.act != kActNone;
  if (OUT_BF16) {
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(a.C) + m * a.ldc + n;
    if (full) {
      uint4* c4 = reinterpret_cast<uint4*>(C);
      if (beta_nz) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 old = c4[q];
          const uint32_t w[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
            v[q * 8 + 2 * e] = fmaf(a.beta, __low2float(h), v[q * 8 + 2 * e]);
            v[q * 8 + 2 * e + 1] = fmaf(a.beta, __high2float(h), v[q * 8 + 2 * e + 1]);
          }
        }
      }
      if (epi) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = finish(a, v[j], n + j);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 o;
        o.x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
        o.y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
        o.z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
        o.w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
        c4[q] = o;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (n + j < a.N) {
          float x = v[j];
          if (beta_nz) x = fmaf(a.beta, __bfloat162float(C[j]), x);
          C[j] = __float2bfloat16_rn(finish(a, x, n + j));
        }
      }
    }
  } else {
    float* C = static_cast<float*>(a.C) + m * a.ldc + n;
    if (full) {
      float4* c4 = reinterpret_cast<float4*>(C);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 o = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        if (beta_nz) {
          const float4 old = c4[q];
          o.x = fmaf(a.beta, old.x, o.x);
          o.y = fmaf(a.beta, old.y, o.y);
          o.z = fmaf(a.beta, old.z, o.z);
          o.w = fmaf(a.beta, old.w, o.w);
        }
        if (epi) {
          o.x = finish(a, o.x, n + 4 * q);
          o.y = finish(a, o.y, n + 4 * q + 1);
          o.z = finish(a, o.z, n + 4 * q + 2);
          o.w = finish(a, o.w, n + 4 * q + 3);
        }
        c4[q] = o;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (n + j < a.N) {
          float x = v[j];
          if (beta_nz) x = fmaf(a.beta, C[j], x);
          C[j] = finish(a, x, n + j);
        }
      }
    }
  }
}

}  // namespace
}  // namespace g3
