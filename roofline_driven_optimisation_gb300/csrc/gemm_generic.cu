// Correctness-first GEMM kernel for any shape, leading dimension and
// (element-aligned) pointer: the path for calls the fast kernels reject.
//
// It is the block-tiled scheme of "CUDA 算子工程 ch.10 朴素 GEMM 与 Roofline
// 分析", sections 10.4-10.6: a 64 x 64 C tile per block, A and B K-slices of
// 16 staged in shared memory (zero-padded outside the matrix, as the bounds
// guards of the thread-tile kernel in 10.6 do), and a 4 x 4 register tile per
// thread.  Accumulation is fp32 for both input types.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "epilogue.cuh"
#include "internal.h"

namespace g3 {
namespace {

constexpr int GT = 64;   // tile edge
constexpr int GK = 16;   // K slice

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// FP8 element (uint8_t) in format fmt (Fp8Fmt): every E4M3 and E5M2 value
// is exact in fp16, so the conversion through fp16 is exact
__device__ __forceinline__ float fp8_to_f32(uint8_t v, int fmt) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(v, fmt == kE5M2 ? __NV_E5M2 : __NV_E4M3);
  return __half2float(__half(h));
}

template <typename T>
__device__ __forceinline__ float load_in(const T* p, long long i, int fmt) {
  if constexpr (std::is_same<T, uint8_t>::value)
    return fp8_to_f32(p[i], fmt);
  else
    return to_f32<T>(p[i]);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// SWIGLU: a second B (a.B2) and accumulator; C = silu(A*B) * (A*B2).
template <typename TI, typename TO, bool SWIGLU>
__global__ void __launch_bounds__(256) gemm_generic_kernel(GemmArgs a, int tiles_n) {
  __shared__ float As[GK][GT + 1];  // As[k][m]
  __shared__ float Bs[GK][GT + 1];  // Bs[k][n]
  __shared__ float Bs2[SWIGLU ? GK : 1][GT + 1];
  const TI* A = static_cast<const TI*>(a.A);
  const TI* B = static_cast<const TI*>(a.B);
  const TI* B2 = static_cast<const TI*>(a.B2);
  TO* C = static_cast<TO*>(a.C);
  const int tile = blockIdx.x;
  const long long m0 = (long long)(tile / tiles_n) * GT;
  const long long n0 = (long long)(tile % tiles_n) * GT;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4], acc2[SWIGLU ? 4 : 1][SWIGLU ? 4 : 1];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  if (SWIGLU) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc2[SWIGLU ? i : 0][SWIGLU ? j : 0] = 0.f;
  }

  for (long long k0 = 0; k0 < a.K; k0 += GK) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int idx = threadIdx.x + r * 256;
      const int am = idx / GK, ak = idx % GK;
      const long long gm = m0 + am, gk = k0 + ak;
      As[ak][am] = (gm < a.M && gk < a.K) ? load_in<TI>(A, gm * a.lda + gk, a.fmt_a) : 0.f;
      const int bk = idx / GT, bn = idx % GT;
      const long long hk = k0 + bk, hn = n0 + bn;
      Bs[bk][bn] = (hk < a.K && hn < a.N) ? load_in<TI>(B, hk * a.ldb + hn, a.fmt_b) : 0.f;
      if (SWIGLU)
        Bs2[SWIGLU ? bk : 0][bn] = (hk < a.K && hn < a.N) ? load_in<TI>(B2, hk * a.ldb + hn, 0) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      if (SWIGLU) {
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Bs2[SWIGLU ? kk : 0][tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            acc2[SWIGLU ? i : 0][SWIGLU ? j : 0] =
                fmaf(av[i], bv[j], acc2[SWIGLU ? i : 0][SWIGLU ? j : 0]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long m = m0 + ty + 16 * i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long n = n0 + tx + 16 * j;
      if (n >= a.N) continue;
      if (SWIGLU) {
        C[m * a.ldc + n] = from_f32<TO>(swiglu_combine(acc[i][j], acc2[SWIGLU ? i : 0][SWIGLU ? j : 0]));
        continue;
      }
      float v = a.alpha * acc[i][j];
      if (a.beta != 0.f) v = fmaf(a.beta, to_f32<TO>(C[m * a.ldc + n]), v);
      C[m * a.ldc + n] = from_f32<TO>(finish(a, v, n));
    }
  }
}

}  // namespace

int launch_generic(const GemmArgs& a, cudaStream_t s) {
  const long long tiles_m = (a.M + GT - 1) / GT;
  const long long tiles_n = (a.N + GT - 1) / GT;
  const long long tiles = tiles_m * tiles_n;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)tiles), block(256);
  if (a.swiglu) {
    if (a.in == Elem::BF16 && a.out == Elem::BF16)
      gemm_generic_kernel<__nv_bfloat16, __nv_bfloat16, true><<<grid, block, 0, s>>>(a, (int)tiles_n);
    else
      return cudaErrorInvalidValue;
  } else if (a.in == Elem::F32 && a.out == Elem::F32) {
    gemm_generic_kernel<float, float, false><<<grid, block, 0, s>>>(a, (int)tiles_n);
  } else if (a.in == Elem::BF16 && a.out == Elem::BF16) {
    gemm_generic_kernel<__nv_bfloat16, __nv_bfloat16, false><<<grid, block, 0, s>>>(a, (int)tiles_n);
  } else if (a.in == Elem::BF16 && a.out == Elem::F32) {
    gemm_generic_kernel<__nv_bfloat16, float, false><<<grid, block, 0, s>>>(a, (int)tiles_n);
  } else if (a.in == Elem::FP8 && a.out == Elem::BF16) {
    gemm_generic_kernel<uint8_t, __nv_bfloat16, false><<<grid, block, 0, s>>>(a, (int)tiles_n);
  } else if (a.in == Elem::FP8 && a.out == Elem::F32) {
    gemm_generic_kernel<uint8_t, float, false><<<grid, block, 0, s>>>(a, (int)tiles_n);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace g3
