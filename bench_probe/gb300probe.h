/*
 * Measurement probe for bench.py and its tests -- C ABI (not part of the GEMM library).
 *
 * The roofline of "Kernel 性能从何而来" (section on the roofline model) bounds
 * a compute-bound kernel by the peak arithmetic rate.  For the FP32 CUDA-core
 * GEMM that peak is SMs x 128 FP32 lanes x 2 FLOP x SM clock; this probe
 * measures what the lanes retire so that the definition can be confirmed on
 * the device, with scalar FMAs and with the packed two-lane fma.rn.f32x2.
 */
#ifndef GB300PROBE_H
#define GB300PROBE_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Launch, on `stream`, a grid of 4 blocks of 256 threads per SM, each thread
 * running 16 independent two-lane FP32 FMA chains for `iters` rounds: packed
 * != 0 issues one fma.rn.f32x2 per chain and round, packed == 0 two scalar
 * FMAs.  The caller times the launch (CUDA events on `stream`).
 *   sink   DEVICE pointer to one float, owned by the caller; written only in
 *          a case that does not occur for these chains (it keeps them live).
 *   flops  HOST pointer; receives the FLOPs of the launch (2 per FMA lane).
 * Returns 0 on success, 1 for iters <= 0 or a NULL pointer, 4 if a CUDA call
 * failed (nothing launched).  Asynchronous; no allocation.
 */
int probe_fp32_fma(int packed, int iters, float* sink, double* flops, cudaStream_t stream);

/*
 * HBM floors for kernels timed alone between two events.
 * probe_read_stream: launches on `stream` a read-only pass over `bytes` bytes
 * of the DEVICE buffer `buf` (16-byte aligned, bytes a multiple of 16) with
 * 16-byte streaming loads, two CTAs of 512 threads per SM.  `sink` is a
 * DEVICE pointer to one unsigned, written only in a case that does not occur
 * for real data (it keeps the loads live).
 * probe_empty: launches one empty CTA on `stream` (the launch alone).
 * Return 0 on success, 1 for bad arguments, 4 if a CUDA call failed.
 * Asynchronous; no allocation.
 */
int probe_read_stream(const void* buf, size_t bytes, unsigned* sink, cudaStream_t stream);
int probe_empty(cudaStream_t stream);

/*
 * Launches on `stream` one CTA that spins on the global timer for `ns`
 * nanoseconds (at most 1e9; larger values return 1) and returns, so the
 * stream stays busy while the host enqueues a batch of timed launches.
 */
int probe_hold(unsigned long long ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300PROBE_H */
