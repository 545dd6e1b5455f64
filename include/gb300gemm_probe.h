/*
 * gb300gemm measurement probe -- C ABI.
 *
 * The roofline of "Kernel 性能从何而来" (section on the roofline model) bounds
 * a compute-bound kernel by the peak arithmetic rate.  For the FP32 CUDA-core
 * GEMM that peak is SMs x 128 FP32 lanes x 2 FLOP x SM clock; this probe
 * measures what the lanes retire so that the definition can be confirmed on
 * the device, with scalar FMAs and with the packed two-lane fma.rn.f32x2.
 */
#ifndef GB300GEMM_PROBE_H
#define GB300GEMM_PROBE_H

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
int gemm_probe_fp32_fma(int packed, int iters, float* sink, double* flops, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300GEMM_PROBE_H */
