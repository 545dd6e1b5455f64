// C ABI of the GEMM library: argument validation, the shape dispatcher, TMA
// tensor-map encoding, and the device status word.
//
// Dispatch (one rule per kernel family):
//   fp32 in/out, TMA-eligible operands           -> register-tiled FP32 kernel
//   bf16 in, M <= 16, TMA-eligible operands       -> split-K skinny kernel
//   bf16 in, M > 16, TMA-eligible operands        -> tcgen05 tensor-core kernel
//   anything else (K == 0, misaligned operands)   -> generic tiled kernel
// The rule follows the roofline classification of "Kernel 性能从何而来"
// ("用 Roofline 指导优化"): a decode-shaped GEMM has an arithmetic intensity
// of about M FLOP/byte and is bandwidth-bound, a large one is compute-bound.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "gb300gemm.h"
#include "internal.h"
#include "ptx.cuh"

namespace g3 {
namespace {

// ---------------------------------------------------------------- errors
thread_local char t_msg[512] = "";
thread_local int t_forced_path = GEMM_PATH_AUTO;
thread_local int t_last_path = GEMM_PATH_AUTO;
thread_local int t_forced_bn = 0;
thread_local int t_last_bn = 0;
thread_local int t_forced_pair = 0;
thread_local int t_last_pair = 0;
thread_local int t_split_tiles = 1;
thread_local int t_last_k_split = 1;
thread_local int t_stall = 0;
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s
constexpr uint64_t kMinTimeoutNs = 1000000ull;         // 1 ms
constexpr uint64_t kMaxTimeoutNs = 10000000000ull;     // 10 s
std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return code;
}

// ---------------------------------------------------------------- devices
__device__ int g_status_word;
// Values taken by gemm_device_status: one slot per call in flight (a host
// counter picks the slot), so concurrent readers on other streams never
// overwrite each other's result.
constexpr int kTakeSlots = 64;
__device__ int g_status_taken[kTakeSlots];

__global__ void status_take_kernel(int* status, int* out) { *out = atomicExch(status, 0); }

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  std::atomic<bool> ready{false};   // published after the fields below are set
  bool supported = false;
  int num_sms = 0;
  int* status = nullptr;
  int* taken = nullptr;   // g_status_taken on this device
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mutex;

int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GEMM_ERR_UNSUPPORTED, "device index %d", dev);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!d.ready.load(std::memory_order_relaxed)) {
      int major = 0, minor = 0, sms = 0;
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return fail(GEMM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
      d.supported = (major == 10 && minor == 3);
      d.num_sms = sms;
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_status_word);
      if (e != cudaSuccess)
        return fail(GEMM_ERR_CUDA, "status word address: %s", cudaGetErrorString(e));
      d.status = static_cast<int*>(p);
      e = cudaGetSymbolAddress(&p, g_status_taken);
      if (e != cudaSuccess)
        return fail(GEMM_ERR_CUDA, "status slot address: %s", cudaGetErrorString(e));
      d.taken = static_cast<int*>(p);
      d.ready.store(true, std::memory_order_release);
    }
  }
  if (!d.supported)
    return fail(GEMM_ERR_UNSUPPORTED, "device %d is not an sm_103 (GB300) GPU", dev);
  *out = &d;
  return GEMM_OK;
}

// ---------------------------------------------------------------- tensor maps
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

struct MapKey {
  uintptr_t ptr;
  uint64_t cols, rows, ld_bytes;
  uint32_t box_cols, box_rows, dtype, swizzle;
  uint64_t depth = 1, ld2_bytes = 0;   // 3-D maps: the third extent and its stride
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && cols == o.cols && rows == o.rows && ld_bytes == o.ld_bytes &&
           box_cols == o.box_cols && box_rows == o.box_rows && dtype == o.dtype &&
           swizzle == o.swizzle && depth == o.depth && ld2_bytes == o.ld2_bytes;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
    h ^= (k.cols + 0x9E37u) * 0xC2B2AE3D27D4EB4Full + (h << 6) + (h >> 2);
    h ^= (k.rows + 0x7F4Au) * 0x165667B19E3779F9ull + (h << 6) + (h >> 2);
    h ^= (k.ld_bytes ^ ((uint64_t)k.box_cols << 32) ^ ((uint64_t)k.box_rows << 48) ^
          ((uint64_t)k.dtype << 8) ^ k.swizzle) * 0x27D4EB2F165667C5ull;
    h ^= (k.depth * 0x9E3779B97F4A7C15ull) ^ (k.ld2_bytes * 0xC2B2AE3D27D4EB4Full);
    return (size_t)h;
  }
};
thread_local std::unordered_map<MapKey, CUtensorMap, MapKeyHash> t_maps;

// The cache is bounded by emptying it at the start of an entry point, never
// inside make_map: a call holds pointers to its earlier maps (A's while B's is
// made), and clearing would leave them dangling.
void trim_maps() {
  if (t_maps.size() > 1024) t_maps.clear();
}

// 2-D row-major matrix (rows x cols, leading dimension ld_bytes) as a TMA
// tensor with box (box_cols x box_rows); elements outside read as zero.
int make_map(const void* ptr, uint64_t cols, uint64_t rows, uint64_t ld_bytes, uint32_t box_cols,
             uint32_t box_rows, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle,
             const CUtensorMap** out) {
  MapKey key{reinterpret_cast<uintptr_t>(ptr), cols, rows, ld_bytes, box_cols, box_rows,
             (uint32_t)dtype, (uint32_t)swizzle};
  auto it = t_maps.find(key);
  if (it != t_maps.end()) {
    *out = &it->second;
    return GEMM_OK;
  }
  EncodeFn fn = encode_fn();
  if (!fn) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap map;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&map, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llux%llu ld=%llu", (int)r,
                (unsigned long long)rows, (unsigned long long)cols, (unsigned long long)ld_bytes);
  auto ins = t_maps.emplace(key, map);
  *out = &ins.first->second;
  return GEMM_OK;
}

// A 3-D tiled map: cols x rows x depth with row stride ld_bytes and depth
// stride ld2_bytes; boxes of box_cols x box_rows x 1.
int make_map_3d(const void* ptr, uint64_t cols, uint64_t rows, uint64_t depth, uint64_t ld_bytes,
                uint64_t ld2_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapDataType dtype,
                CUtensorMapSwizzle swizzle, const CUtensorMap** out) {
  MapKey key{reinterpret_cast<uintptr_t>(ptr), cols, rows, ld_bytes, box_cols, box_rows,
             (uint32_t)dtype, (uint32_t)swizzle, depth, ld2_bytes};
  auto it = t_maps.find(key);
  if (it != t_maps.end()) {
    *out = &it->second;
    return GEMM_OK;
  }
  EncodeFn fn = encode_fn();
  if (!fn) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  CUtensorMap map;
  const cuuint64_t dims[3] = {cols, rows, depth};
  const cuuint64_t strides[2] = {ld_bytes, ld2_bytes};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(&map, dtype, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
  auto ins = t_maps.emplace(key, map);
  *out = &ins.first->second;
  return GEMM_OK;
}

// ---------------------------------------------------------------- dispatch
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// swiglu: C = silu(A*B) * (A*B2), B2 with B's shape and leading dimension
// (alpha 1, beta 0, no bias or activation).
// in == FP8: fmt_a, fmt_b give the 8-bit formats of A and B.
int run(Elem in, Elem out, int M, int N, int K, float alpha, const void* A, int lda, const void* B,
        int ldb, float beta, void* C, int ldc, const float* bias, int act, cudaStream_t stream,
        bool swiglu = false, const void* B2 = nullptr, int fmt_a = kE4M3, int fmt_b = kE4M3) {
  trim_maps();
  t_msg[0] = '\0';
  t_last_path = GEMM_PATH_AUTO;
  t_last_k_split = 1;
  if (M < 0 || N < 0 || K < 0) return fail(GEMM_ERR_INVALID_ARG, "negative size M=%d N=%d K=%d", M, N, K);
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return fail(GEMM_ERR_INVALID_ARG, "leading dimension too small (lda=%d ldb=%d ldc=%d, K=%d N=%d)",
                lda, ldb, ldc, K, N);
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr) return fail(GEMM_ERR_INVALID_ARG, "C is NULL");
  if (K > 0 && (A == nullptr || B == nullptr || (swiglu && B2 == nullptr)))
    return fail(GEMM_ERR_INVALID_ARG, "A or B is NULL");
  const size_t in_sz = in == Elem::F32 ? 4 : in == Elem::BF16 ? 2 : 1;
  const size_t out_sz = out == Elem::F32 ? 4 : 2;
  if (in == Elem::FP8 && (fmt_a < kE4M3 || fmt_a > kE5M2 || fmt_b < kE4M3 || fmt_b > kE5M2))
    return fail(GEMM_ERR_INVALID_ARG, "unknown FP8 format (A %d, B %d)", fmt_a, fmt_b);
  if ((reinterpret_cast<uintptr_t>(A) % in_sz) || (reinterpret_cast<uintptr_t>(B) % in_sz) ||
      (reinterpret_cast<uintptr_t>(B2) % in_sz) || (reinterpret_cast<uintptr_t>(C) % out_sz))
    return fail(GEMM_ERR_MISALIGNED, "a matrix pointer is not aligned to its element size");
  if (act < kActNone || act > kActGelu) return fail(GEMM_ERR_INVALID_ARG, "unknown activation %d", act);
  if (reinterpret_cast<uintptr_t>(bias) % sizeof(float))
    return fail(GEMM_ERR_MISALIGNED, "bias is not aligned to 4 bytes");

  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != GEMM_OK) return rc;
  // the first GEMM call on a device sets up the stream-K workspace, whatever
  // its shape, so that later calls (and stream captures) never allocate
  const cudaError_t we = stream_k_setup(dev->num_sms);
  if (we != cudaSuccess)
    return fail(GEMM_ERR_CUDA, "stream-K workspace: %s", cudaGetErrorString(we));

  GemmArgs a;
  a.M = M; a.N = N; a.K = K; a.alpha = alpha; a.beta = beta;
  a.A = A; a.lda = lda; a.B = B; a.ldb = ldb; a.C = C; a.ldc = ldc;
  a.in = in; a.out = out;
  a.status = dev->status;
  a.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  a.bias = bias;
  a.act = act;
  a.B2 = B2;
  a.swiglu = swiglu ? 1 : 0;
  a.fmt_a = fmt_a;
  a.fmt_b = fmt_b;
  a.stall = t_stall;

  const bool tma_ok = K > 0 && aligned16(A) && aligned16(B) && (!swiglu || aligned16(B2)) &&
                      ((size_t)lda * in_sz) % 16 == 0 && ((size_t)ldb * in_sz) % 16 == 0;
  int path;
  const int forced = t_forced_path;
  if (forced == GEMM_PATH_AUTO) {
    if (!tma_ok) path = GEMM_PATH_GENERIC;
    else if (in == Elem::F32) path = GEMM_PATH_F32_SIMT;
    else if (in == Elem::FP8) path = GEMM_PATH_BF16_TC;
    else if (M <= kSkMaxM) path = GEMM_PATH_SKINNY;
    else path = GEMM_PATH_BF16_TC;
  } else {
    path = forced;
    const bool fits = forced == GEMM_PATH_GENERIC ||
                      (tma_ok && ((forced == GEMM_PATH_F32_SIMT && in == Elem::F32 && !swiglu) ||
                                  (forced == GEMM_PATH_BF16_TC && in != Elem::F32) ||
                                  (forced == GEMM_PATH_SKINNY && in == Elem::BF16 && M <= kSkMaxM)));
    if (!fits) return fail(GEMM_ERR_UNSUPPORTED, "forced path %d cannot run this call", forced);
  }

  int err = cudaSuccess;
  const CUtensorMap *mA = nullptr, *mB = nullptr, *mB2 = nullptr;
  switch (path) {
    case GEMM_PATH_GENERIC:
      err = launch_generic(a, stream);
      break;
    case GEMM_PATH_F32_SIMT: {
      // forced tile widths: 128 -> 8 x 8 register tiles, 256 -> 8 x 16
      if (t_forced_bn != 0 && t_forced_bn != kSimtBN8 && t_forced_bn != kSimtBN16)
        return fail(GEMM_ERR_UNSUPPORTED, "FP32 tiles are 128 or 256 wide, not %d", t_forced_bn);
      SimtPlan plan;
      const int forced_tn = t_forced_bn == kSimtBN16 ? 16 : t_forced_bn == kSimtBN8 ? 8 : 0;
      if ((err = plan_f32_simt(M, N, K, dev->num_sms, forced_tn, &plan)) != cudaSuccess) break;
      if ((rc = make_map(A, K, M, (uint64_t)lda * 4, kSimtBK, kSimtBM, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         CU_TENSOR_MAP_SWIZZLE_64B, &mA)) != GEMM_OK)
        return rc;
      if ((rc = make_map(B, N, K, (uint64_t)ldb * 4, (uint32_t)(16 * plan.tn), kSimtBK,
                         CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE, &mB)) != GEMM_OK)
        return rc;
      err = launch_f32_simt(a, mA, mB, plan, dev->num_sms, stream, &t_last_k_split);
      if (err == cudaSuccess) t_last_bn = 16 * plan.tn;
      break;
    }
    case GEMM_PATH_BF16_TC:
      if (in == Elem::FP8) {
        if ((rc = make_map(A, K, M, (uint64_t)lda, kF8BK, kTcBM, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                           CU_TENSOR_MAP_SWIZZLE_128B, &mA)) != GEMM_OK)
          return rc;
        if ((rc = make_map(B, N, K, (uint64_t)ldb, 128, kF8BK, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                           CU_TENSOR_MAP_SWIZZLE_128B, &mB)) != GEMM_OK)
          return rc;
        int schedule = 2;
        err = launch_fp8_tc_pair(a, mA, mB, dev->num_sms, stream, &schedule);
        if (err == cudaSuccess) {
          t_last_bn = 256;
          t_last_pair = schedule;
        }
        break;
      }
      if ((rc = make_map(A, K, M, (uint64_t)lda * 2, kTcBK, kTcBM, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         CU_TENSOR_MAP_SWIZZLE_128B, &mA)) != GEMM_OK)
        return rc;
      if ((rc = make_map(B, N, K, (uint64_t)ldb * 2, 64, kTcBK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         CU_TENSOR_MAP_SWIZZLE_128B, &mB)) != GEMM_OK)
        return rc;
      if (swiglu) {
        if ((rc = make_map(B2, N, K, (uint64_t)ldb * 2, 64, kTcBK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           CU_TENSOR_MAP_SWIZZLE_128B, &mB2)) != GEMM_OK)
          return rc;
        err = launch_bf16_swiglu_pair(a, mA, mB, mB2, dev->num_sms, stream);
        if (err == cudaSuccess) {
          t_last_bn = 128;  // C columns per tile
          t_last_pair = 2;
        }
        break;
      }
    {
      int pair = 1, bn = 256;
      choose_tc_config(M, N, dev->num_sms, &pair, &bn);
      if (t_forced_bn) {
        bn = t_forced_bn;
        // widths only the single-CTA kernel has imply single CTAs
        if (bn != 128 && bn != 256) pair = 1;
      }
      if (t_forced_pair) pair = t_forced_pair;
      if (pair == 2 && bn != 128 && bn != 256)
        return fail(GEMM_ERR_UNSUPPORTED, "CTA-pair tiles are 128 or 256 wide, not %d", bn);
      int schedule = 1;
      err = pair == 2 ? launch_bf16_tc_pair(a, mA, mB, bn, dev->num_sms, stream, &schedule)
                      : launch_bf16_tc(a, mA, mB, bn, dev->num_sms, stream);
      if (err == cudaSuccess) {
        t_last_bn = bn;
        t_last_pair = schedule;
      }
    }
      break;
    case GEMM_PATH_SKINNY:
      if ((rc = make_map(A, K, M, (uint64_t)lda * 2, kSkBK, kSkMaxM, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         CU_TENSOR_MAP_SWIZZLE_128B, &mA)) != GEMM_OK)
        return rc;
      if ((rc = make_map(B, N, K, (uint64_t)ldb * 2, 64, kSkBK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         CU_TENSOR_MAP_SWIZZLE_128B, &mB)) != GEMM_OK)
        return rc;
      if (swiglu && (rc = make_map(B2, N, K, (uint64_t)ldb * 2, 64, kSkBK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                   CU_TENSOR_MAP_SWIZZLE_128B, &mB2)) != GEMM_OK)
        return rc;
      err = launch_skinny(a, mA, mB, mB2, dev->num_sms, stream, &t_last_k_split);
      break;
    default:
      return fail(GEMM_ERR_INVALID_ARG, "unknown path %d", path);
  }
  if (err != cudaSuccess)
    return fail(GEMM_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString((cudaError_t)err));
  t_last_path = path;
  return GEMM_OK;
}

// A 2-D tensor map encoded into caller storage (no cache: gemm_f32_noalloc
// makes no host allocation either).
int encode_map_into(CUtensorMap* map, const void* ptr, uint64_t cols, uint64_t rows, uint64_t ld_bytes,
                    uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  EncodeFn fn = encode_fn();
  if (!fn) return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llux%llu ld=%llu", (int)r,
                (unsigned long long)rows, (unsigned long long)cols, (unsigned long long)ld_bytes);
  return GEMM_OK;
}

// gemm_f32_noalloc: the FP32 call of run() (no bias or activation) with the
// stream-K tail's scratch in the static array of gemm_f32_simt.cu.  Allocates
// no device or host memory.
int run_f32_noalloc(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                    int ldb, float beta, float* C, int ldc, cudaStream_t stream) {
  t_msg[0] = '\0';
  t_last_path = GEMM_PATH_AUTO;
  t_last_k_split = 1;
  if (M < 0 || N < 0 || K < 0) return fail(GEMM_ERR_INVALID_ARG, "negative size M=%d N=%d K=%d", M, N, K);
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return fail(GEMM_ERR_INVALID_ARG, "leading dimension too small (lda=%d ldb=%d ldc=%d, K=%d N=%d)",
                lda, ldb, ldc, K, N);
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr) return fail(GEMM_ERR_INVALID_ARG, "C is NULL");
  if (K > 0 && (A == nullptr || B == nullptr)) return fail(GEMM_ERR_INVALID_ARG, "A or B is NULL");
  if ((reinterpret_cast<uintptr_t>(A) % 4) || (reinterpret_cast<uintptr_t>(B) % 4) ||
      (reinterpret_cast<uintptr_t>(C) % 4))
    return fail(GEMM_ERR_MISALIGNED, "a matrix pointer is not aligned to its element size");

  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != GEMM_OK) return rc;

  GemmArgs a;
  a.M = M; a.N = N; a.K = K; a.alpha = alpha; a.beta = beta;
  a.A = A; a.lda = lda; a.B = B; a.ldb = ldb; a.C = C; a.ldc = ldc;
  a.in = Elem::F32; a.out = Elem::F32;
  a.status = dev->status;
  a.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  a.bias = nullptr;
  a.act = kActNone;
  a.B2 = nullptr;
  a.swiglu = 0;
  a.fmt_a = kE4M3;
  a.fmt_b = kE4M3;
  a.stall = t_stall;

  const bool tma_ok = K > 0 && aligned16(A) && aligned16(B) && ((size_t)lda * 4) % 16 == 0 &&
                      ((size_t)ldb * 4) % 16 == 0;
  const int forced = t_forced_path;
  if (forced != GEMM_PATH_AUTO && forced != GEMM_PATH_GENERIC &&
      !(forced == GEMM_PATH_F32_SIMT && tma_ok))
    return fail(GEMM_ERR_UNSUPPORTED, "forced path %d cannot run this call", forced);
  int err = cudaSuccess;
  int path = GEMM_PATH_GENERIC;
  if (!tma_ok || forced == GEMM_PATH_GENERIC) {
    err = launch_generic(a, stream);   // no scratch
  } else {
    path = GEMM_PATH_F32_SIMT;
    if (t_forced_bn != 0 && t_forced_bn != kSimtBN8 && t_forced_bn != kSimtBN16)
      return fail(GEMM_ERR_UNSUPPORTED, "FP32 tiles are 128 or 256 wide, not %d", t_forced_bn);
    SimtPlan plan;
    const int forced_tn = t_forced_bn == kSimtBN16 ? 16 : t_forced_bn == kSimtBN8 ? 8 : 0;
    if ((err = plan_f32_simt(M, N, K, dev->num_sms, forced_tn, &plan)) != cudaSuccess)
      return fail(GEMM_ERR_CUDA, "FP32 planning failed: %s", cudaGetErrorString((cudaError_t)err));
    const int ctas = simt_stream_k_ctas(M, N, K, plan, dev->num_sms);
    if (ctas > kStaticScratchCtas)
      return fail(GEMM_ERR_UNSUPPORTED,
                  "gemm_f32_noalloc: the stream-K tail of this %dx%dx%d call needs scratch for %d CTAs "
                  "(%zu bytes); the static scratch holds %d CTAs (%zu bytes): use gemm_f32",
                  M, N, K, ctas, (size_t)ctas * 2 * kSimtBM * kSimtBN16 * sizeof(float),
                  kStaticScratchCtas, simt_static_scratch_bytes());
    CUtensorMap mA, mB;
    if ((rc = encode_map_into(&mA, A, K, M, (uint64_t)lda * 4, kSimtBK, kSimtBM,
                              CU_TENSOR_MAP_SWIZZLE_64B)) != GEMM_OK)
      return rc;
    if ((rc = encode_map_into(&mB, B, N, K, (uint64_t)ldb * 4, (uint32_t)(16 * plan.tn), kSimtBK,
                              CU_TENSOR_MAP_SWIZZLE_NONE)) != GEMM_OK)
      return rc;
    err = launch_f32_simt_static(a, &mA, &mB, plan, dev->num_sms, stream, &t_last_k_split);
    if (err == cudaSuccess) t_last_bn = 16 * plan.tn;
  }
  if (err != cudaSuccess)
    return fail(GEMM_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString((cudaError_t)err));
  t_last_path = path;
  return GEMM_OK;
}

int int4_dequant(const uint8_t* q, int K, int N, int ldq, const void* scales, int lds, int group,
                int zero, void* W, int ldw, bool out_bf16, cudaStream_t stream) {
  t_msg[0] = '\0';
  t_last_path = GEMM_PATH_AUTO;
  t_last_k_split = 1;
  if (K < 0 || N < 0) return fail(GEMM_ERR_INVALID_ARG, "negative size K=%d N=%d", K, N);
  if (group < 1) return fail(GEMM_ERR_INVALID_ARG, "group size %d < 1", group);
  if (zero < 0 || zero > 15) return fail(GEMM_ERR_INVALID_ARG, "zero point %d outside 0..15", zero);
  const int bytes_per_row = (N + 1) / 2;
  if (ldq < (bytes_per_row > 1 ? bytes_per_row : 1) || lds < (N > 1 ? N : 1) || ldw < (N > 1 ? N : 1))
    return fail(GEMM_ERR_INVALID_ARG, "leading dimension too small (ldq=%d lds=%d ldw=%d, N=%d)", ldq,
                lds, ldw, N);
  if (K == 0 || N == 0) return GEMM_OK;
  if (q == nullptr || scales == nullptr || W == nullptr)
    return fail(GEMM_ERR_INVALID_ARG, "q, scales or W is NULL");
  if ((reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(W) & (out_bf16 ? 1u : 3u)))
    return fail(GEMM_ERR_MISALIGNED, "scales or W is not aligned to its element size");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != GEMM_OK) return rc;
  int vec = 0;
  const int err = launch_int4_dequant(q, K, N, ldq, scales, lds, group, zero, W, ldw, out_bf16,
                                      dev->num_sms, stream, &vec);
  if (err != cudaSuccess)
    return fail(GEMM_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString((cudaError_t)err));
  t_last_path = vec ? GEMM_PATH_INT4 : GEMM_PATH_GENERIC;
  return GEMM_OK;
}

int int4_repack(const uint8_t* q, int K, int N, int ldq, uint8_t* qk, cudaStream_t stream) {
  t_msg[0] = '\0';
  t_last_path = GEMM_PATH_AUTO;
  t_last_k_split = 1;
  if (K < 0 || N < 0) return fail(GEMM_ERR_INVALID_ARG, "negative size K=%d N=%d", K, N);
  const int bpr = (N + 1) / 2;
  if (ldq < (bpr > 1 ? bpr : 1))
    return fail(GEMM_ERR_INVALID_ARG, "leading dimension too small (ldq=%d, N=%d)", ldq, N);
  if (K == 0 || N == 0) return GEMM_OK;
  if (q == nullptr || qk == nullptr) return fail(GEMM_ERR_INVALID_ARG, "q or qk is NULL");
  if (reinterpret_cast<uintptr_t>(qk) & 15u) return fail(GEMM_ERR_MISALIGNED, "qk is not 16-byte aligned");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != GEMM_OK) return rc;
  const int err = launch_int4_repack(q, ldq, qk, K, N, dev->num_sms, stream);
  if (err != cudaSuccess)
    return fail(GEMM_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString((cudaError_t)err));
  return GEMM_OK;
}

int w4a16(int M, int N, int K, float alpha, const void* X, int ldx, const uint8_t* qk,
          const void* scales, int lds, int group, int zero, float beta, void* C, int ldc, Elem out,
          cudaStream_t stream) {
  trim_maps();
  t_msg[0] = '\0';
  t_last_path = GEMM_PATH_AUTO;
  t_last_k_split = 1;
  if (M < 0 || N < 0 || K < 0) return fail(GEMM_ERR_INVALID_ARG, "negative size M=%d N=%d K=%d", M, N, K);
  if (group < 1) return fail(GEMM_ERR_INVALID_ARG, "group size %d < 1", group);
  if (zero < 0 || zero > 15) return fail(GEMM_ERR_INVALID_ARG, "zero point %d outside 0..15", zero);
  if (ldx < (K > 1 ? K : 1) || lds < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return fail(GEMM_ERR_INVALID_ARG, "leading dimension too small (ldx=%d lds=%d ldc=%d)", ldx, lds, ldc);
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr) return fail(GEMM_ERR_INVALID_ARG, "C is NULL");
  if (K > 0 && (X == nullptr || qk == nullptr || scales == nullptr))
    return fail(GEMM_ERR_INVALID_ARG, "X, qk or scales is NULL");
  const size_t out_sz = out == Elem::F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(X) & 1u) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (reinterpret_cast<uintptr_t>(C) % out_sz))
    return fail(GEMM_ERR_MISALIGNED, "X, scales or C is not aligned to its element size");
  if (reinterpret_cast<uintptr_t>(qk) & 15u) return fail(GEMM_ERR_MISALIGNED, "qk is not 16-byte aligned");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != GEMM_OK) return rc;
  GemmArgs a{};
  a.M = M; a.N = N; a.K = K; a.alpha = alpha; a.beta = beta;
  a.A = X; a.lda = ldx; a.B = qk; a.ldb = 0; a.C = C; a.ldc = ldc;
  a.in = Elem::BF16; a.out = out;
  a.status = dev->status;
  a.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  a.bias = nullptr; a.act = kActNone; a.B2 = nullptr; a.swiglu = 0; a.fmt_a = 0; a.fmt_b = 0;
  const bool fast = w4_fast_ok(M, K, group) && aligned16(X) && ((size_t)ldx * 2) % 16 == 0 &&
                    t_forced_path != GEMM_PATH_GENERIC;
  const CUtensorMap* mX = nullptr;
  if (fast && (rc = make_map(X, K, M, (uint64_t)ldx * 2, kSkBK, kSkMaxM, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                             CU_TENSOR_MAP_SWIZZLE_128B, &mX)) != GEMM_OK)
    return rc;
  const int err = launch_w4_decode(a, scales, lds, group, zero, mX, qk, fast, dev->num_sms, stream,
                                   &t_last_k_split);
  if (err != cudaSuccess)
    return fail(GEMM_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString((cudaError_t)err));
  t_last_path = fast ? GEMM_PATH_W4 : GEMM_PATH_GENERIC;
  return GEMM_OK;
}

int attention(int B, int Hq, int Hkv, int Sq, int Sk, int D, const void* Q, const void* K, const void* V,
              void* O, float scale, int causal, cudaStream_t stream) {
  trim_maps();
  t_msg[0] = '\0';
  t_last_path = GEMM_PATH_AUTO;
  t_last_k_split = 1;
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Sk < 0 || D < 1)
    return fail(GEMM_ERR_INVALID_ARG, "bad sizes B=%d Hq=%d Hkv=%d Sq=%d Sk=%d D=%d", B, Hq, Hkv, Sq, Sk, D);
  if (Hq > 0 && (Hkv < 1 || Hq % Hkv != 0))
    return fail(GEMM_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (!(scale >= 0.f) || !std::isfinite(scale)) return fail(GEMM_ERR_INVALID_ARG, "bad scale");
  if (B == 0 || Hq == 0 || Sq == 0) return GEMM_OK;
  // one grid row per (batch, head): the grid's y extent is at most 65535
  if ((long long)B * Hq > 65535)
    return fail(GEMM_ERR_UNSUPPORTED, "B*Hq = %lld exceeds 65535 (batch x heads)", (long long)B * Hq);
  if (Q == nullptr || O == nullptr || (Sk > 0 && (K == nullptr || V == nullptr)))
    return fail(GEMM_ERR_INVALID_ARG, "Q, K, V or O is NULL");
  if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) |
       reinterpret_cast<uintptr_t>(O)) & 1u)
    return fail(GEMM_ERR_MISALIGNED, "a tensor is not aligned to 2 bytes");
  if (((size_t)Sk + 32) * 4 > 227 * 1024 && !(D == 64 || D == 128))
    return fail(GEMM_ERR_UNSUPPORTED, "Sk %d too long for the generic attention kernel", Sk);
  if (scale == 0.f) scale = 1.f / std::sqrt((float)D);
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc != GEMM_OK) return rc;
  const bool fast = (D == 64 || D == 128) && Sk > 0 && aligned16(Q) && aligned16(K) && aligned16(V) &&
                    aligned16(O) && t_forced_path != GEMM_PATH_GENERIC;
  if (!fast && ((size_t)Sk + 32) * 4 > 227 * 1024)
    return fail(GEMM_ERR_UNSUPPORTED, "Sk %d too long for the generic attention kernel", Sk);
  const CUtensorMap *mQ = nullptr, *mK = nullptr, *mV = nullptr;
  if (fast) {
    const uint64_t row = (uint64_t)D * 2;
    if ((rc = make_map_3d(Q, D, Sq, (uint64_t)B * Hq, row, row * Sq, 64, 128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          CU_TENSOR_MAP_SWIZZLE_128B, &mQ)) != GEMM_OK)
      return rc;
    if ((rc = make_map_3d(K, D, Sk, (uint64_t)B * Hkv, row, row * Sk, 64, 64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          CU_TENSOR_MAP_SWIZZLE_128B, &mK)) != GEMM_OK)
      return rc;
    if ((rc = make_map_3d(V, D, Sk, (uint64_t)B * Hkv, row, row * Sk, 64, 64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          CU_TENSOR_MAP_SWIZZLE_128B, &mV)) != GEMM_OK)
      return rc;
  }
  const int err = launch_attention(B, Hq, Hkv, Sq, Sk, D, Q, K, V, O, scale, causal ? 1 : 0, mQ, mK, mV, fast,
                                   dev->status, g_timeout_ns.load(std::memory_order_relaxed), stream);
  if (err != cudaSuccess)
    return fail(GEMM_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString((cudaError_t)err));
  t_last_path = fast ? GEMM_PATH_ATTN : GEMM_PATH_GENERIC;
  return GEMM_OK;
}

__global__ void selftest_wait_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait must run out.
  if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, timeout_ns, nullptr))
    report_status(status, GEMM_ERR_DEVICE_TIMEOUT, kSiteSelftest);
}

}  // namespace

bool split_tiles_enabled() { return t_split_tiles != 0; }
int split_tiles_mode() { return t_split_tiles; }

}  // namespace g3

using g3::Elem;

extern "C" {

int gemm_f32(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
             float beta, float* C, int ldc, cudaStream_t stream) {
  return g3::run(Elem::F32, Elem::F32, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr,
                 g3::kActNone, stream);
}

int gemm_f32_noalloc(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                     int ldb, float beta, float* C, int ldc, cudaStream_t stream) {
  return g3::run_f32_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

int gemm_bf16(int M, int N, int K, float alpha, const gemm_bf16_t* A, int lda, const gemm_bf16_t* B,
              int ldb, float beta, gemm_bf16_t* C, int ldc, cudaStream_t stream) {
  return g3::run(Elem::BF16, Elem::BF16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr,
                 g3::kActNone, stream);
}

int gemm_bf16_f32out(int M, int N, int K, float alpha, const gemm_bf16_t* A, int lda,
                     const gemm_bf16_t* B, int ldb, float beta, float* C, int ldc,
                     cudaStream_t stream) {
  return g3::run(Elem::BF16, Elem::F32, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr,
                 g3::kActNone, stream);
}

int gemm_bf16_swiglu(int M, int N, int K, const gemm_bf16_t* A, int lda, const gemm_bf16_t* Bgate,
                     const gemm_bf16_t* Bup, int ldb, gemm_bf16_t* C, int ldc, cudaStream_t stream) {
  return g3::run(Elem::BF16, Elem::BF16, M, N, K, 1.f, A, lda, Bgate, ldb, 0.f, C, ldc, nullptr,
                 g3::kActNone, stream, /*swiglu=*/true, Bup);
}

int gemm_fp8(int M, int N, int K, float alpha, const uint8_t* A, int fmt_a, int lda, const uint8_t* B,
             int fmt_b, int ldb, float beta, gemm_bf16_t* C, int ldc, cudaStream_t stream) {
  return g3::run(Elem::FP8, Elem::BF16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr,
                 g3::kActNone, stream, false, nullptr, fmt_a, fmt_b);
}

int gemm_fp8_f32out(int M, int N, int K, float alpha, const uint8_t* A, int fmt_a, int lda,
                    const uint8_t* B, int fmt_b, int ldb, float beta, float* C, int ldc,
                    cudaStream_t stream) {
  return g3::run(Elem::FP8, Elem::F32, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr,
                 g3::kActNone, stream, false, nullptr, fmt_a, fmt_b);
}

int gemm_int4_dequant(const uint8_t* q, int K, int N, int ldq, const gemm_bf16_t* scales, int lds,
                      int group, int zero, gemm_bf16_t* W, int ldw, cudaStream_t stream) {
  return g3::int4_dequant(q, K, N, ldq, scales, lds, group, zero, W, ldw, true, stream);
}

int gemm_int4_dequant_f32(const uint8_t* q, int K, int N, int ldq, const gemm_bf16_t* scales,
                          int lds, int group, int zero, float* W, int ldw, cudaStream_t stream) {
  return g3::int4_dequant(q, K, N, ldq, scales, lds, group, zero, W, ldw, false, stream);
}

int gemm_attention(int B, int Hq, int Hkv, int Sq, int Sk, int D, const gemm_bf16_t* Q, const gemm_bf16_t* K,
                   const gemm_bf16_t* V, gemm_bf16_t* O, float scale, int causal, cudaStream_t stream) {
  return g3::attention(B, Hq, Hkv, Sq, Sk, D, Q, K, V, O, scale, causal, stream);
}

size_t gemm_w4_packed_bytes(int K, int N) { return g3::w4_packed_bytes(K, N); }

int gemm_int4_repack(const uint8_t* q, int K, int N, int ldq, uint8_t* qk, cudaStream_t stream) {
  return g3::int4_repack(q, K, N, ldq, qk, stream);
}

int gemm_w4a16(int M, int N, int K, float alpha, const gemm_bf16_t* X, int ldx, const uint8_t* qk,
               const gemm_bf16_t* scales, int lds, int group, int zero, float beta, gemm_bf16_t* C,
               int ldc, cudaStream_t stream) {
  return g3::w4a16(M, N, K, alpha, X, ldx, qk, scales, lds, group, zero, beta, C, ldc, Elem::BF16,
                   stream);
}

int gemm_w4a16_f32out(int M, int N, int K, float alpha, const gemm_bf16_t* X, int ldx,
                      const uint8_t* qk, const gemm_bf16_t* scales, int lds, int group, int zero,
                      float beta, float* C, int ldc, cudaStream_t stream) {
  return g3::w4a16(M, N, K, alpha, X, ldx, qk, scales, lds, group, zero, beta, C, ldc, Elem::F32,
                   stream);
}

int gemm_f32_ex(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
                float beta, float* C, int ldc, const float* bias, int activation,
                cudaStream_t stream) {
  return g3::run(Elem::F32, Elem::F32, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias,
                 activation, stream);
}

int gemm_bf16_ex(int M, int N, int K, float alpha, const gemm_bf16_t* A, int lda,
                 const gemm_bf16_t* B, int ldb, float beta, gemm_bf16_t* C, int ldc,
                 const float* bias, int activation, cudaStream_t stream) {
  return g3::run(Elem::BF16, Elem::BF16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias,
                 activation, stream);
}

int gemm_bf16_f32out_ex(int M, int N, int K, float alpha, const gemm_bf16_t* A, int lda,
                        const gemm_bf16_t* B, int ldb, float beta, float* C, int ldc,
                        const float* bias, int activation, cudaStream_t stream) {
  return g3::run(Elem::BF16, Elem::F32, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias,
                 activation, stream);
}

const char* gemm_get_last_error(void) { return g3::t_msg; }

int gemm_device_status(cudaStream_t stream, int* where) {
  if (where) *where = 0;
  g3::DeviceInfo* dev = nullptr;
  int rc = g3::device_info(&dev);
  if (rc != GEMM_OK) return rc;
  // One atomic exchange on the device takes the word and leaves it zero: a
  // failure recorded by a kernel on any stream is either in this value or
  // stays for the next call, never lost between a read and a clear.
  static std::atomic<unsigned> next_slot{0};
  int* slot = dev->taken + (next_slot.fetch_add(1, std::memory_order_relaxed) % g3::kTakeSlots);
  g3::status_take_kernel<<<1, 1, 0, stream>>>(dev->status, slot);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return g3::fail(GEMM_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  int word = 0;
  e = cudaMemcpyAsync(&word, slot, sizeof(word), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return g3::fail(GEMM_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
  if (where) *where = (int)((unsigned)word >> 8);
  // a kernel that gave up may have left stream-K flags raised: lower them
  // before the workspace is used again
  if ((word & 0xff) == GEMM_ERR_DEVICE_TIMEOUT) g3::sk_clear_flags();
  return word & 0xff;
}

int gemm_force_path(int path) {
  if (path < GEMM_PATH_AUTO || path > GEMM_PATH_SKINNY)
    return g3::fail(GEMM_ERR_INVALID_ARG, "unknown path %d", path);
  g3::t_forced_path = path;
  return GEMM_OK;
}

int gemm_last_path(void) { return g3::t_last_path; }

int gemm_force_tile_n(int bn) {
  if (bn != 0 && bn != 128 && bn != 192 && bn != 224 && bn != 256)
    return g3::fail(GEMM_ERR_INVALID_ARG, "tile width %d is not 0, 128, 192, 224 or 256", bn);
  g3::t_forced_bn = bn;
  return GEMM_OK;
}

int gemm_last_tile_n(void) { return g3::t_last_bn; }

int gemm_force_tc_pair(int mode) {
  if (mode < 0 || mode > 2) return g3::fail(GEMM_ERR_INVALID_ARG, "pair mode %d is not 0, 1 or 2", mode);
  g3::t_forced_pair = mode;
  return GEMM_OK;
}

int gemm_last_tc_pair(void) { return g3::t_last_pair; }

int gemm_force_split_tiles(int enable) {
  if (enable < 0 || enable > 3) return g3::fail(GEMM_ERR_INVALID_ARG, "enable must be 0, 1, 2 or 3");
  g3::t_split_tiles = enable;
  return GEMM_OK;
}

int gemm_last_k_split(void) { return g3::t_last_k_split; }

int gemm_set_wait_timeout_ns(uint64_t timeout_ns) {
  if (timeout_ns == 0) timeout_ns = g3::kDefaultTimeoutNs;
  if (timeout_ns < g3::kMinTimeoutNs || timeout_ns > g3::kMaxTimeoutNs)
    return g3::fail(GEMM_ERR_INVALID_ARG, "timeout_ns %llu outside [1e6, 1e10] (0 = default 1e9)",
                    (unsigned long long)timeout_ns);
  g3::g_timeout_ns.store(timeout_ns);
  return GEMM_OK;
}

int gemm_test_stall(int enable) {
  if (enable != 0 && enable != 1) return g3::fail(GEMM_ERR_INVALID_ARG, "enable must be 0 or 1");
  g3::t_stall = enable;
  return GEMM_OK;
}

int gemm_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
  if (timeout_ns == 0 || timeout_ns > 1000000000ull)
    return g3::fail(GEMM_ERR_INVALID_ARG, "timeout_ns must be in (0, 1e9]");
  g3::DeviceInfo* dev = nullptr;
  int rc = g3::device_info(&dev);
  if (rc != GEMM_OK) return rc;
  g3::selftest_wait_kernel<<<1, 32, 0, stream>>>(dev->status, timeout_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return g3::fail(GEMM_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return GEMM_OK;
}

}  // extern "C"
