/*
 * gb300gemm -- dense GEMM for NVIDIA GB300 (sm_103a), C ABI.
 *
 * Every entry point computes
 *
 *     C = alpha * A * B + beta * C
 *
 * the general matrix multiply of "CUDA 算子工程, ch.10 朴素 GEMM 与 Roofline
 * 分析", section 10.1 (the GEMM equation), on row-major matrices as indexed by
 * the naive kernel of section 10.2 (A[row*K + k], B[k*N + col],
 * C[row*N + col]), with explicit leading dimensions:
 *
 *     A is M x K, element (i, k) at A[i*lda + k], lda >= K
 *     B is K x N, element (k, j) at B[k*ldb + j], ldb >= N
 *     C is M x N, element (i, j) at C[i*ldc + j], ldc >= N
 *
 * Conventions shared by all GEMM entry points
 *   - All matrix pointers are DEVICE pointers owned by the caller; the library
 *     never frees or retains them past the call.  A and B are read only.
 *   - Products are accumulated in fp32; the epilogue alpha*acc + beta*C is
 *     evaluated in fp32 and rounded once (round-to-nearest-even) to C's type.
 *   - beta == 0 makes C write-only: the old C is never read, so NaN or Inf
 *     there does not reach the result.
 *   - M == 0 or N == 0 is a no-op.  K == 0 gives C = beta*C.
 *   - The call is asynchronous on `stream` (0 = legacy default stream).  It
 *     performs no host synchronisation and no device allocation, except the
 *     first GEMM call (gemm_f32*, gemm_bf16*, gemm_fp8*) on a device: it
 *     allocates the stream-K workspace that the FP32 SIMT and CTA-pair
 *     tensor-core kernels share (four slots of 39.8 MB of partial tiles on
 *     152 SMs, plus flags; kept until the process exits), zeroes its flags
 *     and waits for the device once.
 *   - Fast paths need 16-byte-aligned A and B and lda, ldb whose byte size is
 *     a multiple of 16; anything else still runs, on a generic GPU kernel.
 *     There is no CPU fallback.
 *   - Results of one call are deterministic: the same inputs give the same
 *     bits on every run (fixed reduction order, including split-K).
 *   - Calls made concurrently from several host threads are safe.  Calls
 *     whose partial last wave runs stream-K (FP32: gemm_last_k_split() > 1
 *     on a wide tile; tensor core: gemm_last_tc_pair() == 6) take the four
 *     workspace slots in turn: at most four of them may execute on the GPU
 *     at the same time (on different streams, or in graphs launched side by
 *     side); a fifth would share a slot with the first and race with it.
 *   - Calls can be captured into a CUDA graph (stream capture) once the same
 *     kind of call has run on the device: the first call of a kernel family
 *     on a device sets kernel attributes and queries occupancy.
 *
 * Errors: every entry point returns a gemm_status.  On a non-zero return
 * nothing was launched (except when the second launch of a two-launch call,
 * the FP32 path's split last wave, fails after the first was queued) and
 * gemm_get_last_error() describes the cause.  Errors
 * found on the device (a bounded wait that ran out) are recorded in a status
 * word that gemm_device_status() reads.
 */
#ifndef GB300GEMM_H
#define GB300GEMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
#include <cuda_bf16.h>
typedef __nv_bfloat16 gemm_bf16_t;
extern "C" {
#else
typedef uint16_t gemm_bf16_t; /* IEEE bfloat16 bit pattern */
#endif

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1,   /* negative size, ld too small, null pointer */
  GEMM_ERR_MISALIGNED = 2,    /* pointer not aligned to its element size */
  GEMM_ERR_UNSUPPORTED = 3,   /* size beyond the supported range, no sm_103a device */
  GEMM_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (message has its text) */
  GEMM_ERR_DEVICE_TIMEOUT = 5 /* a kernel's bounded wait ran out (device status only) */
} gemm_status;

/*
 * FP32 SGEMM on the CUDA cores ("CUDA 算子工程 ch.10", sections 10.4-10.6:
 * block tile in shared memory, warp tile, register tile).
 * A, B, C: fp32.  alpha, beta: fp32.
 */
int gemm_f32(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
             float beta, float* C, int ldc, cudaStream_t stream);

/*
 * gemm_f32 for callers that must not allocate.  The source pages have no
 * counterpart of this entry point: it is a library addition.
 *
 * Who needs it: a caller that hands the device's memory to its own pool up
 * front (a caching allocator that reserves nearly all of it, or a process
 * under a fixed memory budget) cannot let a library allocate later -- the
 * allocation may fail, or break the pool's accounting; and a caller on a
 * latency-critical thread cannot take the device-wide wait that the first
 * GEMM call of the other entry points makes on a device while it sets up
 * the stream-K workspace.
 *
 * Same arguments, result and error codes as gemm_f32, the same plan and
 * the same kernels (so the same bits for the same inputs).  The one
 * difference: when the plan runs the last partial wave as a stream-K tail,
 * its partial tiles and flags live in a static device array of this library
 * (38 MiB of partial tiles plus 9.5 KB of flags, reserved on each device
 * when the FP32 kernel's module loads), not in an allocated workspace.  The
 * call allocates no device or host memory and performs no host
 * synchronisation.
 *
 * Limit: the array holds the tail of at most 152 CTAs (one per SM of a
 * GB300).  A call whose tail would need more (a device with more SMs)
 * returns GEMM_ERR_UNSUPPORTED, launches nothing, and gemm_get_last_error()
 * states the bytes needed and held.
 *
 * Set-up: the first call on a device (with that device current) looks up
 * the array's device address; make that first call before any stream
 * capture.  Each call with a stream-K tail first clears the array's flags
 * on `stream`.
 *
 * Concurrency: there is one array per device, so two gemm_f32_noalloc calls
 * that execute on one device at the same time (on different streams, with
 * nothing ordering them) race and may both give wrong results.  Order them
 * on one stream or with events.  gemm_f32 calls do not share the array.
 */
int gemm_f32_noalloc(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                     int ldb, float beta, float* C, int ldc, cudaStream_t stream);

/*
 * BF16 GEMM with fp32 accumulation and bf16 C, on the tensor cores
 * (tcgen05.mma fed by TMA, "Kernel 性能从何而来", section "优化阶梯").  Small M
 * (decode-shaped, M <= 16) runs on a memory-bound split-K kernel instead
 * (same page, section "优化 Memory-Bound Kernel").
 * A, B, C: bf16.  alpha, beta: fp32.
 */
int gemm_bf16(int M, int N, int K, float alpha, const gemm_bf16_t* A, int lda,
              const gemm_bf16_t* B, int ldb, float beta, gemm_bf16_t* C, int ldc,
              cudaStream_t stream);

/*
 * As gemm_bf16, but C is fp32 (read when beta != 0, written always).
 */
int gemm_bf16_f32out(int M, int N, int K, float alpha, const gemm_bf16_t* A, int lda,
                     const gemm_bf16_t* B, int ldb, float beta, float* C, int ldc,
                     cudaStream_t stream);

/* Activation applied last by the _ex entry points. */
typedef enum {
  GEMM_ACT_NONE = 0,
  GEMM_ACT_RELU = 1, /* max(z, 0) */
  GEMM_ACT_SILU = 2, /* z / (1 + exp(-z)) */
  GEMM_ACT_GELU = 3  /* 0.5 z (1 + erf(z / sqrt(2))) */
} gemm_activation;

/*
 * The three GEMMs with a fused elementwise epilogue ("Kernel 性能从何而来",
 * section "优化 Memory-Bound Kernel": fuse the GEMM with its elementwise
 * epilogue instead of a second pass over C):
 *
 *     z = alpha * A*B + beta * C + bias      (bias[n] added to every row m)
 *     C = act(z)
 *
 * z and act(z) are evaluated in fp32 and rounded once to C's type.  `bias` is
 * a DEVICE pointer to N floats (4-byte aligned) or NULL; `activation` is a
 * gemm_activation.  Everything else is as for the plain entry points, which
 * are these with bias = NULL and GEMM_ACT_NONE.
 */
int gemm_f32_ex(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
                float beta, float* C, int ldc, const float* bias, int activation,
                cudaStream_t stream);
int gemm_bf16_ex(int M, int N, int K, float alpha, const gemm_bf16_t* A, int lda,
                 const gemm_bf16_t* B, int ldb, float beta, gemm_bf16_t* C, int ldc,
                 const float* bias, int activation, cudaStream_t stream);
int gemm_bf16_f32out_ex(int M, int N, int K, float alpha, const gemm_bf16_t* A, int lda,
                        const gemm_bf16_t* B, int ldb, float beta, float* C, int ldc,
                        const float* bias, int activation, cudaStream_t stream);

/*
 * The FFN gate/up pair of a LLaMA layer ("CUDA 算子工程 ch.10 朴素 GEMM 与
 * Roofline 分析", section 10.1: FFN gate / up / down as separate GEMMs, SiLU
 * among the small elementwise operators) fused into one kernel, as
 * "Kernel 性能从何而来" section "优化 Memory-Bound Kernel" asks of a producer
 * and its consumer (the intermediate stays in TMEM/registers):
 *
 *     C = silu(A * Bgate) .* (A * Bup),   silu(z) = z / (1 + exp(-z))
 *
 * A is M x K (lda), Bgate and Bup are K x N with the same leading dimension
 * ldb, C is M x N (ldc); all bf16 DEVICE pointers owned by the caller.  Both
 * products are accumulated in fp32, combined in fp32 and rounded once to
 * bf16.  C is write-only.  K == 0 gives C = 0.  Bup may be NULL only when
 * K == 0.  Alignment, paths, asynchrony, determinism and errors are as for
 * gemm_bf16: M <= 16 runs on the decode kernel, larger M on CTA pairs with
 * 256 x 128 C tiles, unaligned operands on the generic kernel.
 */
int gemm_bf16_swiglu(int M, int N, int K, const gemm_bf16_t* A, int lda, const gemm_bf16_t* Bgate,
                     const gemm_bf16_t* Bup, int ldb, gemm_bf16_t* C, int ldc, cudaStream_t stream);

/* 8-bit floating-point formats of the FP8 entry points (the OCP FP8 formats). */
typedef enum {
  GEMM_FP8_E4M3 = 0, /* 4 exponent bits (bias 7), 3 mantissa bits, no inf, max 448 */
  GEMM_FP8_E5M2 = 1  /* 5 exponent bits (bias 15), 2 mantissa bits, IEEE-like, max 57344 */
} gemm_fp8_format;

/*
 * FP8 GEMM ("Kernel 性能从何而来", section "优化 Memory-Bound Kernel": fp8
 * inputs move fewer bytes per FLOP than fp16 or fp32):
 *
 *     C = alpha * A * B + beta * C
 *
 * A is M x K and B is K x N, one byte per element, each in its own format
 * (fmt_a, fmt_b: gemm_fp8_format), row-major with leading dimensions lda >= K
 * and ldb >= N in elements (= bytes).  Per-tensor scale factors of a
 * quantised layer fold into alpha.  The products are exact and accumulated
 * in fp32, and the epilogue is that of gemm_bf16: bf16 C (gemm_fp8) or fp32 C
 * (gemm_fp8_f32out).  The fast path runs on CTA pairs with 256 x 256 C tiles
 * (tcgen05 kind::f8f6f4).  It needs 16-byte-aligned A and B, and lda and ldb
 * multiples of 16.  Anything else runs on the generic kernel.  Conventions,
 * errors and asynchrony are those of gemm_bf16.  An unknown format returns
 * GEMM_ERR_INVALID_ARG.
 */
int gemm_fp8(int M, int N, int K, float alpha, const uint8_t* A, int fmt_a, int lda, const uint8_t* B,
             int fmt_b, int ldb, float beta, gemm_bf16_t* C, int ldc, cudaStream_t stream);
int gemm_fp8_f32out(int M, int N, int K, float alpha, const uint8_t* A, int fmt_a, int lda,
                    const uint8_t* B, int fmt_b, int ldb, float beta, float* C, int ldc,
                    cudaStream_t stream);

/*
 * INT4 weight dequantisation ("CUDA 算子工程 ch.4 内存层级与代价表", section
 * 4.5.3: two 4-bit codes per byte, the first in the low nibble, times a
 * scale):
 *
 *     W[k][n] = scales[k / group][n] * (q[k][n] - zero)
 *
 * q is K x N codes (0..15) packed along n: byte j of row k (row stride ldq
 * bytes, ldq >= ceil(N/2)) holds column 2j in bits 0-3 and column 2j+1 in
 * bits 4-7.  scales is ceil(K/group) x N bf16 (row stride lds >= N elements).
 * zero is one integer in 0..15, and group >= 1.  W is K x N (ldw >= N),
 * written as bf16 by gemm_int4_dequant (the exact fp32 value rounded once,
 * nearest even) or as fp32 by gemm_int4_dequant_f32 (exact).  All pointers
 * are DEVICE pointers owned by the caller.  The fastest kernel (a thread
 * per 4, 8 or 16 rows of 8 or 4 columns) needs N a multiple of 8, K and
 * group both multiples of 4, 4-byte-aligned rows of q and 16-byte-aligned
 * rows of scales and W; the next needs N a multiple of 32 and 16-byte-
 * aligned rows of all three.  Other shapes run a per-byte kernel.  All give
 * the same bits.  Errors and asynchrony are as for the GEMM entry points.
 */
int gemm_int4_dequant(const uint8_t* q, int K, int N, int ldq, const gemm_bf16_t* scales, int lds,
                      int group, int zero, gemm_bf16_t* W, int ldw, cudaStream_t stream);
int gemm_int4_dequant_f32(const uint8_t* q, int K, int N, int ldq, const gemm_bf16_t* scales,
                          int lds, int group, int zero, float* W, int ldw, cudaStream_t stream);

/*
 * INT4 weight-only decode GEMM ("CUDA 算子工程 ch.4 内存层级与代价表",
 * section 4.5.3, dequantisation fused into its consumer as "Kernel 性能从何而来"
 * section "优化 Memory-Bound Kernel" asks):
 *
 *     C = alpha * X * W + beta * C,   W[k][n] = scales[k / group][n] * (q[k][n] - zero)
 *
 * X is M x K bf16 (ldx >= K), C is M x N (ldc >= N), bf16 (gemm_w4a16) or
 * fp32 (gemm_w4a16_f32out), scales and zero as for gemm_int4_dequant.  The
 * weight is the exact value: the products take the integers q - zero and each
 * group's fp32 sum is multiplied by its scale, so W is never rounded.  qk holds
 * the codes in the tiled layout that gemm_int4_repack writes
 * (gemm_w4_packed_bytes(K, N) bytes, 16-byte aligned).  beta == 0 never reads
 * C.  The fast path is the tcgen05 decode kernel.  It needs 1 <= M <= 16,
 * group a multiple of 64 or group >= K, and X 16-byte aligned with ldx a
 * multiple of 8.  Any other call runs a one-thread-per-element kernel.
 * Conventions, errors, determinism and asynchrony are those of the GEMM entry
 * points.
 */
int gemm_w4a16(int M, int N, int K, float alpha, const gemm_bf16_t* X, int ldx, const uint8_t* qk,
               const gemm_bf16_t* scales, int lds, int group, int zero, float beta, gemm_bf16_t* C,
               int ldc, cudaStream_t stream);
int gemm_w4a16_f32out(int M, int N, int K, float alpha, const gemm_bf16_t* X, int ldx,
                      const uint8_t* qk, const gemm_bf16_t* scales, int lds, int group, int zero,
                      float beta, float* C, int ldc, cudaStream_t stream);

/*
 * The tiled INT4 layout of gemm_w4a16.  W is cut into tiles of 128 columns
 * by 64 rows of K, 4 KB each, stored column tiles outer and K tiles inner.
 * Inside a tile, column n has 32 bytes: eight little-endian 32-bit words, word j
 * packing the codes of k = 8j + 0, 2, 4, 6, 1, 3, 5, 7 in its nibbles 0..7.
 * Tiles and codes past N or K are 0.  gemm_w4_packed_bytes gives the size,
 * ceil(N/128) * ceil(K/64) * 4096 bytes (0 for an empty weight).
 * gemm_int4_repack writes it from the codes of gemm_int4_dequant (K x N,
 * packed along n, ldq bytes per row) into qk (16-byte aligned DEVICE
 * memory of that size).  Done once per weight.
 */
size_t gemm_w4_packed_bytes(int K, int N);
int gemm_int4_repack(const uint8_t* q, int K, int N, int ldq, uint8_t* qk, cudaStream_t stream);

/*
 * Attention forward ("从模型计算到 GPU 执行：读懂算子、Kernel 与 GPU 性能", section
 * 1.2: S = Q K^T, S = S / sqrt(d), P = softmax(S), O = P V), with S and P
 * kept on chip ("Kernel 性能从何而来", section on attention):
 *
 *     O = softmax(Q K^T * scale) V,   per batch b and query head h
 *
 * Q and O are [B][Hq][Sq][D] and K, V are [B][Hkv][Sk][D], all contiguous bf16
 * DEVICE tensors owned by the caller.  Hq must be a multiple of Hkv: query
 * head h reads key/value head h / (Hq / Hkv).  scale == 0 means 1/sqrt(D).
 * causal != 0 lets query i see key j only when j <= i + (Sk - Sq).  Masked
 * scores are -inf, and a row with no visible key gives O = 0.  The softmax
 * is in fp32 (running maximum and sum), P is rounded to bf16 for the second
 * product, and O is rounded once to bf16.  The fast path (tcgen05) needs
 * D = 64 or 128 and 16-byte-aligned tensors.  Other calls run a
 * one-block-per-row kernel, for Sk up to about 58,000.  B * Hq above 65535
 * returns GEMM_ERR_UNSUPPORTED (one grid row per batch and head).  Errors
 * and asynchrony are as for the GEMM entry points.
 */
int gemm_attention(int B, int Hq, int Hkv, int Sq, int Sk, int D, const gemm_bf16_t* Q, const gemm_bf16_t* K,
                   const gemm_bf16_t* V, gemm_bf16_t* O, float scale, int causal, cudaStream_t stream);

/*
 * Message for the last non-OK return on the calling host thread ("" if none).
 * The string is owned by the library and valid until the next call on this
 * thread.
 */
const char* gemm_get_last_error(void);

/*
 * Takes the device status word of the current device: a one-thread kernel on
 * `stream` exchanges it with zero atomically, then the stream is
 * synchronised and the value returned.  The word is per device and shared by
 * every stream and host thread: a failure recorded by a kernel on another
 * stream is either in the value taken or left for the next call, never lost.
 * Returns GEMM_OK, GEMM_ERR_DEVICE_TIMEOUT (a kernel gave up a bounded wait
 * and returned early; its C is unspecified), or GEMM_ERR_CUDA if the launch
 * or synchronisation itself failed.  If `where` is not NULL it receives the
 * kernel-specific location code of the first failure (0 if none).  The
 * `where` argument is this library's addition to the surveyed
 * gemm_device_status(stream); NULL is accepted.
 * When it returns GEMM_ERR_DEVICE_TIMEOUT it also lowers every flag of the
 * device's stream-K workspace (a call that gave up may have left flags
 * raised), with a device-wide memset: take a timeout status while no other
 * stream-K call (see gemm_force_split_tiles) is executing on the device, or
 * that call may report a timeout of its own.
 */
int gemm_device_status(cudaStream_t stream, int* where);

/* Kernel families, for gemm_last_path() and gemm_force_path(). */
typedef enum {
  GEMM_PATH_AUTO = 0,     /* shape dispatcher (default) */
  GEMM_PATH_GENERIC = 1,  /* correctness-first tiled kernel, any alignment */
  GEMM_PATH_F32_SIMT = 2, /* register-tiled FP32 kernel */
  GEMM_PATH_BF16_TC = 3,  /* tcgen05/TMEM/TMA warp-specialised kernel (bf16 or FP8 inputs) */
  GEMM_PATH_SKINNY = 4,   /* decode-shaped split-K kernel (bf16, M <= 16) */
  GEMM_PATH_INT4 = 5,     /* INT4 dequantisation, vector kernel (reported only;
                             the per-byte fallback reports GEMM_PATH_GENERIC) */
  GEMM_PATH_W4 = 6,       /* INT4-weight decode GEMM, tcgen05 kernel (reported only;
                             its one-thread-per-element fallback reports GEMM_PATH_GENERIC) */
  GEMM_PATH_ATTN = 7      /* attention, tcgen05 kernel (reported only; its
                             one-block-per-row fallback reports GEMM_PATH_GENERIC) */
} gemm_path;

/*
 * Pin the kernel family for later calls on this host thread (GEMM_PATH_AUTO
 * restores the dispatcher).  A forced path that cannot run the call (wrong
 * element type, misalignment, M too large for the skinny kernel) makes that
 * call return GEMM_ERR_UNSUPPORTED.  For A/B measurements and tests.
 */
int gemm_force_path(int path);

/* Kernel family the last successful call on this host thread launched
 * (GEMM_PATH_AUTO if it launched nothing). */
int gemm_last_path(void);

/*
 * Pin the C tile width for later calls on this host thread: 128, 192, 224
 * or 256 columns (tiles are 128 rows high); 0 restores the automatic choice,
 * which minimises the work of the last partial wave of tiles over the SMs.
 * The tensor-core kernel takes every width; the FP32 SIMT kernel takes 128
 * (8 x 8 register tiles, two CTAs per SM) or 256 (8 x 16 register tiles, one
 * CTA per SM), and an FP32 call with another forced width returns
 * GEMM_ERR_UNSUPPORTED.  Other values return GEMM_ERR_INVALID_ARG.  For A/B
 * measurements and tests.
 */
int gemm_force_tile_n(int bn);

/* Tile width the last tensor-core or FP32 SIMT call on this host thread used
 * (0 if none). */
int gemm_last_tile_n(void);

/*
 * Pin how the tensor-core kernel maps C tiles to SMs for later calls on this
 * host thread: 1 = one CTA per 128-row tile, 2 = a pair of CTAs (a cluster of
 * two issuing one 256-row tcgen05 MMA) per 256-row tile, 0 = automatic.  With
 * 2 only tile widths 128 and 256 exist; a forced width of 192 or 224 makes
 * the call return GEMM_ERR_UNSUPPORTED (with 0 such a width selects single
 * CTAs).  For A/B measurements and tests.
 */
int gemm_force_tc_pair(int mode);

/* For the last tensor-core call on this host thread: 1 if it ran on single
 * CTAs, 2 on CTA pairs, 4 on CTA pairs with the tiles of the last partial
 * wave split into half-width tiles, 6 on CTA pairs with those tiles run
 * stream-K, 0 if there was none. */
int gemm_last_tc_pair(void);

/*
 * Allow (1, the default) or forbid (0), for later calls on this host thread,
 * that the tiles of a partial last wave run split.  The CTA-pair kernel's
 * 256-wide tiles run them either as two half-width tiles each on otherwise
 * idle pairs (bf16 only) or stream-K: the tail's K-steps spread evenly over
 * the pairs, each tile's partial sums added by one pair in pair order; a
 * wave model picks one.  The FP32 SIMT kernel runs them as a second launch
 * in which a cluster of four CTAs shares each tile's K range (partial sums
 * added in rank order, in distributed shared memory) on its narrow tiles,
 * or stream-K on its wide tiles (the K-slices over up to one CTA per SM).
 * 2 pins the CTA-pair kernel's stream-K tail and 3 its half-width tail
 * wherever the shape has a partial wave (and, for 3, the half tiles fit in
 * the pairs); the FP32 kernel treats 2 and 3 as 1.  Stream-K partial tiles
 * meet in the device's stream-K workspace.  For A/B measurements and tests.
 */
int gemm_force_split_tiles(int enable);

/* For the last call on this host thread: the number of CTAs that shared the
 * K range of one C tile (the decode kernels' cluster split; 4 when the FP32
 * SIMT kernel split its narrow tiles' partial last wave; for its stream-K
 * tail, the most CTAs that met in one tile), 1 if none did. */
int gemm_last_k_split(void);

/*
 * Upper bound, in nanoseconds, on any single wait inside a kernel launched
 * later by this process (default 1e9).  After it a kernel records
 * GEMM_ERR_DEVICE_TIMEOUT in the status word and returns.  0 restores the
 * default; other values outside [1e6, 1e10] (1 ms to 10 s) return
 * GEMM_ERR_INVALID_ARG and leave the bound unchanged.  The waits that let
 * copies and MMAs already in flight land after such an abort have their own
 * fixed bound (200 ms) and do not use this one.
 */
int gemm_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * Test hook for the abort paths of the CTA-pair tensor-core kernel, the
 * decode split-K kernel and the FP32 SIMT kernel (including its split last
 * wave).  With enable = 1, later calls on this host thread make one role of
 * the first CTA or cluster wait on a barrier that nothing arrives at: the MMA
 * issuer of the first pair, the MMA issuer of rank 0 of the first decode
 * cluster, warp 0 of the first FP32 CTA.  That bounded wait runs out after
 * a quarter of the gemm_set_wait_timeout_ns() limit (before any wait that
 * follows from it, so its location code is the one recorded), the kernel records
 * GEMM_ERR_DEVICE_TIMEOUT with that role's location code and leaves through
 * its abort path (the other CTAs of the cluster included); C is unspecified.
 * enable = 0 (the default) turns it off; other values return
 * GEMM_ERR_INVALID_ARG.  Never faults: no copy is skipped and nothing is
 * read or written out of bounds.
 */
int gemm_test_stall(int enable);

/*
 * Self-test of the bounded-wait mechanism: launches one CTA that waits on a
 * shared-memory barrier nothing ever arrives at, with the given bound, then
 * returns.  Afterwards gemm_device_status() reports GEMM_ERR_DEVICE_TIMEOUT.
 * timeout_ns must be in (0, 1e9].
 */
int gemm_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GB300GEMM_H */
