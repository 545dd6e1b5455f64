"""CPU oracle for dense GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it.

* :func:`gemm` is the plain fp64 definition of ``C = alpha*A*B + beta*C0``
  ("CUDA 算子工程 ch.10 朴素 GEMM 与 Roofline 分析", section 10.1), computed by
  ``oracle.c`` (a triple loop over rows, k and columns, k summed in order).
* :func:`normwise_error` is the score the GPU result is held to:
  ``max|C_gpu - C_ref| / max_{m,n} sum_k |A[m,k]| |B[k,n]|``, the denominator
  being the same oracle GEMM applied to |A| and |B|
  (:func:`abs_product_max`).  For alpha != 1 or beta != 0 the scale of the
  whole expression, ``max(|alpha| sum_k |A||B| + |beta| |C0|)``, is used
  (:func:`normwise_denominator`); it equals the former at alpha=1, beta=0.
  For the fused epilogue act(z) the scale is that of z (with |bias|): the
  activations have slope at most 1.13, so an error in z carries over at that
  size.
* ``oracle.epilogue`` holds the activations and the SwiGLU pair.
* ``oracle.roofline_ref`` restates the FLOP, arithmetic-intensity and roofline
  formulas of the pages.

Inputs are numpy/torch arrays holding exactly the values the GPU receives
(fp32 as is, bf16 already rounded); they are widened to fp64 exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into liboracle.so (plain C, no CUDA)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_gemm.argtypes = [
                ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                dp, ctypes.c_long, dp, ctypes.c_long,
                ctypes.c_double, dp, ctypes.c_long, dp, ctypes.c_long, ctypes.c_int]
            lib.oracle_gemm.restype = ctypes.c_int
            _lib = lib
    return _lib


def to_f64(x) -> np.ndarray:
    """Exact widening of an fp32/bf16/fp64 torch tensor or numpy array to fp64."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float64)
    import torch  # local: the oracle itself needs only numpy
    return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def gemm(A, B, alpha: float = 1.0, beta: float = 0.0, C0=None,
         threads: int | None = None) -> np.ndarray:
    """fp64 ``alpha*A@B + beta*C0`` (C0 ignored and unread when beta == 0)."""
    A64 = to_f64(A)
    B64 = to_f64(B)
    if A64.ndim != 2 or B64.ndim != 2 or A64.shape[1] != B64.shape[0]:
        raise ValueError(f"shape mismatch {A64.shape} x {B64.shape}")
    M, K = A64.shape
    N = B64.shape[1]
    R = np.empty((M, N), dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    c0_ptr = None
    c0 = None
    if beta != 0.0:
        if C0 is None:
            raise ValueError("beta != 0 needs C0")
        c0 = to_f64(C0)
        if c0.shape != (M, N):
            raise ValueError("C0 shape")
        c0_ptr = c0.ctypes.data_as(dp)
    if M == 0 or N == 0:
        return R
    lib = _load()
    # numpy gives a valid (non-null) pointer even for K == 0 arrays
    a_ptr = A64.ctypes.data_as(dp) if A64.size else ctypes.cast(R.ctypes.data, dp)
    b_ptr = B64.ctypes.data_as(dp) if B64.size else ctypes.cast(R.ctypes.data, dp)
    rc = lib.oracle_gemm(M, N, K, float(alpha), a_ptr, max(K, 1), b_ptr, N,
                         float(beta), c0_ptr, N, R.ctypes.data_as(dp), N,
                         int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with code {rc}")
    return R


def abs_product_max(A, B, threads: int | None = None) -> float:
    """max_{m,n} sum_k |A[m,k]| |B[k,n]| (the normwise-error denominator)."""
    A64 = np.abs(to_f64(A))
    B64 = np.abs(to_f64(B))
    if A64.shape[0] == 0 or B64.shape[1] == 0:
        return 0.0
    P = gemm(A64, B64, 1.0, 0.0, None, threads)
    return float(P.max()) if P.size else 0.0


def normwise_denominator(A, B, alpha: float = 1.0, beta: float = 0.0, C0=None,
                         threads: int | None = None, bias=None) -> float:
    """max_{m,n} (|alpha| sum_k |A[m,k]||B[k,n]| + |beta| |C0[m,n]|).

    The normwise scale of the whole expression alpha*A*B + beta*C0.  With
    alpha = 1 and beta = 0 it is exactly max sum_k |A||B|; with beta != 0 the
    rounding of C to its output type is relative to |C|, which includes
    beta*C0, so the C0 term belongs in the scale.
    """
    A64 = np.abs(to_f64(A))
    B64 = np.abs(to_f64(B))
    M, N = A64.shape[0], B64.shape[1]
    if M == 0 or N == 0:
        return 0.0
    if beta != 0.0:
        c0 = np.abs(to_f64(C0))
        P = gemm(A64, B64, abs(alpha), abs(beta), c0, threads)
    else:
        P = gemm(A64, B64, abs(alpha), 0.0, None, threads)
    if bias is not None:
        # the fused epilogue's bias is one more term of z = alpha*AB + beta*C0 + bias
        P = P + np.abs(to_f64(bias)).reshape(1, -1)
    return float(P.max())


def normwise_error(C_gpu, C_ref: np.ndarray, denom: float) -> float:
    """max|C_gpu - C_ref| / denom; NaN anywhere in C_gpu gives +inf."""
    G = to_f64(C_gpu)
    if G.shape != C_ref.shape:
        raise ValueError(f"shape mismatch {G.shape} vs {C_ref.shape}")
    if G.size == 0:
        return 0.0
    if not np.all(np.isfinite(G)) and np.all(np.isfinite(C_ref)):
        return float("inf")
    num = float(np.max(np.abs(G - C_ref)))
    if denom == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / denom


# Tolerances on the normwise error, per output type of the path.
TOL_F32 = 1e-5          # gemm_f32
TOL_BF16_OUT = 4e-3     # bf16 inputs, bf16 C
TOL_BF16_F32OUT = 1e-5  # bf16 inputs, fp32 C
