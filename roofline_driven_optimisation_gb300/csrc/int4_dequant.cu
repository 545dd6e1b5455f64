// INT4 weight dequantisation: W[k][n] = s[k / G][n] * (q[k][n] - z), written
// as bf16 (one rounding of the exact fp32 value) or as fp32 (exact).
//
// "CUDA 算子工程 ch.4 内存层级与代价表", section 4.5.3, measures this kernel:
// reading one packed byte per thread is instruction-bound (256 GB/s on its
// GPU), reading 16 bytes (32 codes) per thread and expanding them in
// registers with vector stores reaches 2.1 TB/s.  That layout still reads a
// scale (2 bytes) from L2 for every weight it writes, and each warp store
// instruction covers its 2 KB in 16-byte pieces.  Here a thread takes R rows
// of one column octet (bf16) or quad (fp32): the scales of those columns are
// loaded once for the R rows (R divides the group size), the R code words
// are loaded together, and every warp store writes 512 contiguous bytes.
// fp32 stores carry the evict-first hint.  Calls whose K or group size R
// does not divide, or whose rows are not aligned, run the 32-codes-per-thread
// kernel or a per-byte kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace g3 {
namespace {

constexpr int THREADS = 256;
constexpr int UNROLL = 4;

// fp32 (code - zero) for the two codes of a byte, exact: the magic-number
// float 2^23 + c has c in its low mantissa bits
__device__ __forceinline__ float code_lo(uint32_t word, int byte) {
  return __uint_as_float(0x4B000000u | ((word >> (8 * byte)) & 0xFu)) - 8388608.f;
}
__device__ __forceinline__ float code_hi(uint32_t word, int byte) {
  return __uint_as_float(0x4B000000u | ((word >> (8 * byte + 4)) & 0xFu)) - 8388608.f;
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(THREADS) int4_dequant_vec(const uint8_t* __restrict__ q, long long ldq,
                                                            const __nv_bfloat16* __restrict__ s,
                                                            long long lds, int group, int zero,
                                                            void* __restrict__ w, long long ldw,
                                                            int chunks, long long items) {
  const long long stride = (long long)gridDim.x * THREADS;
  const float fz = (float)zero;
  for (long long base = (long long)blockIdx.x * THREADS + threadIdx.x; base < items;
       base += stride * UNROLL) {
    uint4 pk[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const long long it = base + u * stride;
      if (it < items) {
        const long long k = it / chunks, c = it % chunks;
        pk[u] = __ldcs(reinterpret_cast<const uint4*>(q + k * ldq + c * 16));
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const long long it = base + u * stride;
      if (it >= items) break;
      const long long k = it / chunks, c = it % chunks;
      const uint4* sp = reinterpret_cast<const uint4*>(s + (k / group) * lds + c * 32);
      const uint32_t words[4] = {pk[u].x, pk[u].y, pk[u].z, pk[u].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {          // 8 columns per word of codes
        const uint4 sv = __ldg(sp + h);       // their 8 scales
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
        float v[8];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float s0 = __uint_as_float(sw[b] << 16), s1 = __uint_as_float(sw[b] & 0xFFFF0000u);
          v[2 * b] = s0 * (code_lo(words[h], b) - fz);
          v[2 * b + 1] = s1 * (code_hi(words[h], b) - fz);
        }
        if (OUT_BF16) {
          uint4 o;
          o.x = pack2_bf16(v[0], v[1]);
          o.y = pack2_bf16(v[2], v[3]);
          o.z = pack2_bf16(v[4], v[5]);
          o.w = pack2_bf16(v[6], v[7]);
          __stcs(reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(w) + k * ldw + c * 32 + h * 8), o);
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(w) + k * ldw + c * 32 + h * 8);
          __stcs(dst, make_float4(v[0], v[1], v[2], v[3]));
          __stcs(dst + 1, make_float4(v[4], v[5], v[6], v[7]));
        }
      }
    }
  }
}

// One octet = 8 consecutive columns of one row: 4 bytes of codes, 8 scales
// (16 bytes), 16 or 32 bytes of output.  Consecutive threads take
// consecutive octets, so a warp reads 128 contiguous bytes of codes and
// writes 512 (bf16) or 1024 (fp32) contiguous bytes per instruction.
template <bool OUT_BF16, int UNR>
__global__ void __launch_bounds__(THREADS) int4_dequant_octets(const uint8_t* __restrict__ q, long long ldq,
                                                            const __nv_bfloat16* __restrict__ s,
                                                            long long lds, int group, int zero,
                                                            void* __restrict__ w, long long ldw,
                                                            int octets, long long items) {
  const long long stride = (long long)gridDim.x * THREADS;
  const float fz = (float)zero;
  for (long long base = (long long)blockIdx.x * THREADS + threadIdx.x; base < items;
       base += stride * UNR) {
    uint32_t pk[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const long long it = base + u * stride;
      if (it < items) {
        const long long k = it / octets, o = it % octets;
        pk[u] = __ldcs(reinterpret_cast<const unsigned int*>(q + k * ldq + o * 4));
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const long long it = base + u * stride;
      if (it >= items) break;
      const long long k = it / octets, o = it % octets;
      const uint4 sv = __ldg(reinterpret_cast<const uint4*>(s + (k / group) * lds + o * 8));
      const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
      float v[8];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float s0 = __uint_as_float(sw[b] << 16), s1 = __uint_as_float(sw[b] & 0xFFFF0000u);
        v[2 * b] = s0 * (code_lo(pk[u], b) - fz);
        v[2 * b + 1] = s1 * (code_hi(pk[u], b) - fz);
      }
      if (OUT_BF16) {
        uint4 ov;
        ov.x = pack2_bf16(v[0], v[1]);
        ov.y = pack2_bf16(v[2], v[3]);
        ov.z = pack2_bf16(v[4], v[5]);
        ov.w = pack2_bf16(v[6], v[7]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(w) + k * ldw + o * 8) = ov;
      } else {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(w) + k * ldw + o * 8);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
}

// R consecutive rows of one column octet per thread.  The octet's 8 scales
// are loaded once for the R rows (R divides the group size, so the rows share
// them), the R code words are loaded together, and each row is one 16-byte
// (bf16) or 32-byte (fp32) store.  A warp covers 32 consecutive octets, so
// every load and store instruction of a warp touches contiguous memory, and
// the scales cost 2/R bytes of L2 traffic per weight instead of 2.
template <bool OUT_BF16, int R>
__global__ void __launch_bounds__(THREADS) int4_dequant_rows(const uint8_t* __restrict__ q, long long ldq,
                                                            const __nv_bfloat16* __restrict__ s,
                                                            long long lds, int group, int zero,
                                                            void* __restrict__ w, long long ldw,
                                                            int octets, long long items) {
  const long long stride = (long long)gridDim.x * THREADS;
  // (2^23 + c) - (2^23 + z) = c - z exactly, one subtraction per code
  const float fz = 8388608.f + (float)zero;
  for (long long it = (long long)blockIdx.x * THREADS + threadIdx.x; it < items; it += stride) {
    const long long k0 = (it / octets) * R;
    const int o = (int)(it % octets);
    const uint8_t* qp = q + k0 * ldq + (long long)o * 4;
    uint32_t pk[R];
#pragma unroll
    for (int r = 0; r < R; ++r) pk[r] = __ldcs(reinterpret_cast<const unsigned int*>(qp + r * ldq));
    const uint4 sv = __ldg(reinterpret_cast<const uint4*>(s + (k0 / group) * lds + (long long)o * 8));
    const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
    float sc[8];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      sc[2 * b] = __uint_as_float(sw[b] << 16);
      sc[2 * b + 1] = __uint_as_float(sw[b] & 0xFFFF0000u);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float v[8];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        v[2 * b] = sc[2 * b] * (__uint_as_float(0x4B000000u | ((pk[r] >> (8 * b)) & 0xFu)) - fz);
        v[2 * b + 1] = sc[2 * b + 1] * (__uint_as_float(0x4B000000u | ((pk[r] >> (8 * b + 4)) & 0xFu)) - fz);
      }
      const long long off = (k0 + r) * ldw + (long long)o * 8;
      if (OUT_BF16) {
        uint4 ov;
        ov.x = pack2_bf16(v[0], v[1]);
        ov.y = pack2_bf16(v[2], v[3]);
        ov.z = pack2_bf16(v[4], v[5]);
        ov.w = pack2_bf16(v[6], v[7]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(w) + off) = ov;
      } else {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(w) + off);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
}

// fp32 output: R consecutive rows of one column quad (4 columns, 2 bytes of
// codes, 8 bytes of scales) per thread, so that one warp store instruction
// writes 512 contiguous bytes; the stores are evict-first (nothing rereads
// W from L2 here).
template <int R>
__global__ void __launch_bounds__(THREADS) int4_dequant_rows_f32(const uint8_t* __restrict__ q, long long ldq,
                                                                const __nv_bfloat16* __restrict__ s,
                                                                long long lds, int group, int zero,
                                                                float* __restrict__ w, long long ldw,
                                                                int quads, long long items) {
  const long long stride = (long long)gridDim.x * THREADS;
  const float fz = 8388608.f + (float)zero;
  for (long long it = (long long)blockIdx.x * THREADS + threadIdx.x; it < items; it += stride) {
    const long long k0 = (it / quads) * R;
    const int o = (int)(it % quads);
    const uint8_t* qp = q + k0 * ldq + (long long)o * 2;
    uint32_t pk[R];
#pragma unroll
    for (int r = 0; r < R; ++r) pk[r] = __ldcs(reinterpret_cast<const unsigned short*>(qp + r * ldq));
    const uint2 sv = __ldg(reinterpret_cast<const uint2*>(s + (k0 / group) * lds + (long long)o * 4));
    const float sc[4] = {__uint_as_float(sv.x << 16), __uint_as_float(sv.x & 0xFFFF0000u),
                         __uint_as_float(sv.y << 16), __uint_as_float(sv.y & 0xFFFF0000u)};
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float4 v;
      v.x = sc[0] * (__uint_as_float(0x4B000000u | (pk[r] & 0xFu)) - fz);
      v.y = sc[1] * (__uint_as_float(0x4B000000u | ((pk[r] >> 4) & 0xFu)) - fz);
      v.z = sc[2] * (__uint_as_float(0x4B000000u | ((pk[r] >> 8) & 0xFu)) - fz);
      v.w = sc[3] * (__uint_as_float(0x4B000000u | ((pk[r] >> 12) & 0xFu)) - fz);
      float4* dst = reinterpret_cast<float4*>(w + (k0 + r) * ldw + (long long)o * 4);
      __stcs(dst, v);
    }
  }
}

// one byte (two columns; the high nibble of a last odd column is padding)
template <bool OUT_BF16>
__global__ void __launch_bounds__(THREADS) int4_dequant_bytes(const uint8_t* __restrict__ q, long long ldq,
                                                              const __nv_bfloat16* __restrict__ s,
                                                              long long lds, int group, int zero,
                                                              void* __restrict__ w, long long ldw, int N,
                                                              int bytes_per_row, long long items) {
  const long long stride = (long long)gridDim.x * THREADS;
  for (long long it = (long long)blockIdx.x * THREADS + threadIdx.x; it < items; it += stride) {
    const long long k = it / bytes_per_row, j = it % bytes_per_row;
    const uint32_t b = q[k * ldq + j];
    const __nv_bfloat16* srow = s + (k / group) * lds;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const long long n = 2 * j + e;
      if (n >= N) break;
      const float code = (float)((b >> (4 * e)) & 0xFu);
      const float v = __bfloat162float(srow[n]) * (code - (float)zero);
      if (OUT_BF16)
        static_cast<__nv_bfloat16*>(w)[k * ldw + n] = __float2bfloat16_rn(v);
      else
        static_cast<float*>(w)[k * ldw + n] = v;
    }
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int launch_int4_dequant(const uint8_t* q, int K, int N, int ldq, const void* scales, int lds,
                        int group, int zero, void* w, int ldw, bool out_bf16, int num_sms,
                        cudaStream_t st, int* vector_path) {
  const auto* s = static_cast<const __nv_bfloat16*>(scales);
  const int osz = out_bf16 ? 2 : 4;
  const bool w_ok = al16(s) && lds % 8 == 0 && al16(w) && ((long long)ldw * osz) % 16 == 0;
  const bool vec = out_bf16 ? (w_ok && N % 32 == 0 && al16(q) && ldq % 16 == 0)
                            : (w_ok && N % 8 == 0 && (reinterpret_cast<uintptr_t>(q) & 3u) == 0 &&
                               ldq % 4 == 0);
  *vector_path = vec ? 1 : 0;
  const unsigned grid = (unsigned)num_sms * (2048 / THREADS);
  // rows per thread: the largest of 16, 8, 4 that divides K and the group
  int R = 0;
  for (int r : {16, 8, 4})
    if (!R && K % r == 0 && group % r == 0) R = r;
  const bool rows = R > 0 && N % 8 == 0 && w_ok && (reinterpret_cast<uintptr_t>(q) & 3u) == 0 &&
                    ldq % 4 == 0;
  if (rows) {
    *vector_path = 1;
    if (out_bf16) {
      const int octets = N / 8;
      const long long items = (long long)(K / R) * octets;
      auto* kern = R == 16 ? int4_dequant_rows<true, 16> : R == 8 ? int4_dequant_rows<true, 8>
                                                                  : int4_dequant_rows<true, 4>;
      kern<<<grid, THREADS, 0, st>>>(q, ldq, s, lds, group, zero, w, ldw, octets, items);
    } else {
      const int quads = N / 4;
      const long long items = (long long)(K / R) * quads;
      auto* kern = R == 16 ? int4_dequant_rows_f32<16> : R == 8 ? int4_dequant_rows_f32<8>
                                                                : int4_dequant_rows_f32<4>;
      kern<<<grid, THREADS, 0, st>>>(q, ldq, s, lds, group, zero, static_cast<float*>(w), ldw, quads, items);
    }
  } else if (vec && out_bf16) {
    const int chunks = N / 32;
    const long long items = (long long)K * chunks;
    int4_dequant_vec<true><<<grid, THREADS, 0, st>>>(q, ldq, s, lds, group, zero, w, ldw, chunks, items);
  } else if (vec) {
    const int octets = N / 8;
    const long long items = (long long)K * octets;
    int4_dequant_octets<false, 8><<<grid, THREADS, 0, st>>>(q, ldq, s, lds, group, zero, w, ldw, octets,
                                                            items);
  } else {
    const int bpr = (N + 1) / 2;
    const long long items = (long long)K * bpr;
    if (out_bf16)
      int4_dequant_bytes<true><<<grid, THREADS, 0, st>>>(q, ldq, s, lds, group, zero, w, ldw, N, bpr, items);
    else
      int4_dequant_bytes<false><<<grid, THREADS, 0, st>>>(q, ldq, s, lds, group, zero, w, ldw, N, bpr, items);
  }
  return cudaGetLastError();
}

}  // namespace g3
