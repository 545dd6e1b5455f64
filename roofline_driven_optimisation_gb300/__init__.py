"""GB300 dense GEMM: Python binding of the C-ABI library ``libgb300gemm.so``.

The binding only marshals arguments (device pointers, sizes, leading
dimensions, the CUDA stream handle) to the C entry points declared in
``include/gb300gemm.h``; every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is missing or cannot
be loaded, every call raises.

Low-level calls (same names and argument order as the C ABI; pointers and the
stream are integers):

    gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)
    gemm_bf16(...), gemm_bf16_f32out(...)

Tensor convenience wrapper (reads pointers, strides and the current stream):

    gemm(A, B, C, alpha=1.0, beta=0.0)
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_MISALIGNED = 2
GEMM_ERR_UNSUPPORTED = 3
GEMM_ERR_CUDA = 4
GEMM_ERR_DEVICE_TIMEOUT = 5

PATH_AUTO, PATH_GENERIC, PATH_F32_SIMT, PATH_BF16_TC, PATH_SKINNY, PATH_INT4, PATH_W4, PATH_ATTN = range(8)
ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU = range(4)
FP8_E4M3, FP8_E5M2 = 0, 1
PATH_NAMES = {PATH_AUTO: "none", PATH_GENERIC: "generic", PATH_F32_SIMT: "f32_simt",
              PATH_BF16_TC: "bf16_tc", PATH_SKINNY: "skinny", PATH_INT4: "int4", PATH_W4: "w4",
              PATH_ATTN: "attention"}

# every symbol the public header declares
EXPORTS = ("gemm_f32", "gemm_f32_noalloc", "gemm_bf16", "gemm_bf16_f32out", "gemm_f32_ex", "gemm_bf16_ex",
           "gemm_bf16_f32out_ex", "gemm_bf16_swiglu", "gemm_fp8", "gemm_fp8_f32out",
           "gemm_int4_dequant", "gemm_int4_dequant_f32", "gemm_w4a16", "gemm_w4a16_f32out",
           "gemm_int4_repack", "gemm_w4_packed_bytes", "gemm_attention", "gemm_get_last_error",
           "gemm_device_status", "gemm_force_path", "gemm_last_path", "gemm_force_tile_n",
           "gemm_last_tile_n", "gemm_force_tc_pair", "gemm_last_tc_pair", "gemm_force_split_tiles",
           "gemm_last_k_split", "gemm_set_wait_timeout_ns",
           "gemm_selftest_wait_timeout", "gemm_test_stall")

_lib = None
_lock = threading.Lock()


class GemmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"gemm error {code}: {message}")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    return _build.build(force=force)


def load(path: str | None = None):
    """Load the C library (built in-tree by ``build()``) and declare signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA GEMM library not built: {p} (run __graft_entry__.build())")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        for name in ("gemm_f32", "gemm_f32_noalloc", "gemm_bf16", "gemm_bf16_f32out"):
            fn = getattr(lib, name)
            fn.argtypes = [i, i, i, f, vp, i, vp, i, f, vp, i, vp]
            fn.restype = i
        for name in ("gemm_f32_ex", "gemm_bf16_ex", "gemm_bf16_f32out_ex"):
            fn = getattr(lib, name)
            fn.argtypes = [i, i, i, f, vp, i, vp, i, f, vp, i, vp, i, vp]
            fn.restype = i
        lib.gemm_bf16_swiglu.argtypes = [i, i, i, vp, i, vp, vp, i, vp, i, vp]
        lib.gemm_bf16_swiglu.restype = i
        for name in ("gemm_int4_dequant", "gemm_int4_dequant_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, i, i, i, vp, i, i, i, vp, i, vp]
            fn.restype = i
        for name in ("gemm_w4a16", "gemm_w4a16_f32out"):
            fn = getattr(lib, name)
            fn.argtypes = [i, i, i, f, vp, i, vp, vp, i, i, i, f, vp, i, vp]
            fn.restype = i
        lib.gemm_int4_repack.argtypes = [vp, i, i, i, vp, vp]
        lib.gemm_int4_repack.restype = i
        lib.gemm_attention.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, f, i, vp]
        lib.gemm_attention.restype = i
        lib.gemm_w4_packed_bytes.argtypes = [i, i]
        lib.gemm_w4_packed_bytes.restype = ctypes.c_size_t
        for name in ("gemm_fp8", "gemm_fp8_f32out"):
            fn = getattr(lib, name)
            fn.argtypes = [i, i, i, f, vp, i, i, vp, i, i, f, vp, i, vp]
            fn.restype = i
        lib.gemm_get_last_error.argtypes = []
        lib.gemm_get_last_error.restype = ctypes.c_char_p
        lib.gemm_device_status.argtypes = [vp, ctypes.POINTER(i)]
        lib.gemm_device_status.restype = i
        lib.gemm_force_path.argtypes = [i]
        lib.gemm_force_path.restype = i
        lib.gemm_last_path.argtypes = []
        lib.gemm_last_path.restype = i
        lib.gemm_force_tile_n.argtypes = [i]
        lib.gemm_force_tile_n.restype = i
        lib.gemm_last_tile_n.argtypes = []
        lib.gemm_last_tile_n.restype = i
        lib.gemm_force_tc_pair.argtypes = [i]
        lib.gemm_force_tc_pair.restype = i
        lib.gemm_last_tc_pair.argtypes = []
        lib.gemm_last_tc_pair.restype = i
        lib.gemm_force_split_tiles.argtypes = [i]
        lib.gemm_force_split_tiles.restype = i
        lib.gemm_last_k_split.argtypes = []
        lib.gemm_last_k_split.restype = i
        lib.gemm_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.gemm_set_wait_timeout_ns.restype = i
        lib.gemm_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.gemm_selftest_wait_timeout.restype = i
        lib.gemm_test_stall.argtypes = [i]
        lib.gemm_test_stall.restype = i
        _lib = lib
        return lib


def _check(rc: int):
    if rc != GEMM_OK:
        msg = _lib.gemm_get_last_error().decode(errors="replace")
        raise GemmError(rc, msg)


def gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
    _check(load().gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream))


def gemm_f32_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
    _check(load().gemm_f32_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream))


def gemm_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
    _check(load().gemm_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream))


def gemm_bf16_f32out(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0):
    _check(load().gemm_bf16_f32out(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream))


def gemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act, stream=0):
    _check(load().gemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act, stream))


def gemm_bf16_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act, stream=0):
    _check(load().gemm_bf16_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act, stream))


def gemm_bf16_f32out_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act, stream=0):
    _check(load().gemm_bf16_f32out_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act,
                                      stream))


def gemm_bf16_swiglu(M, N, K, A, lda, Bgate, Bup, ldb, C, ldc, stream=0):
    _check(load().gemm_bf16_swiglu(M, N, K, A, lda, Bgate, Bup, ldb, C, ldc, stream))


def gemm_fp8(M, N, K, alpha, A, fmt_a, lda, B, fmt_b, ldb, beta, C, ldc, stream=0):
    _check(load().gemm_fp8(M, N, K, alpha, A, fmt_a, lda, B, fmt_b, ldb, beta, C, ldc, stream))


def gemm_fp8_f32out(M, N, K, alpha, A, fmt_a, lda, B, fmt_b, ldb, beta, C, ldc, stream=0):
    _check(load().gemm_fp8_f32out(M, N, K, alpha, A, fmt_a, lda, B, fmt_b, ldb, beta, C, ldc,
                                  stream))


def gemm_int4_dequant(q, K, N, ldq, scales, lds, group, zero, W, ldw, stream=0):
    _check(load().gemm_int4_dequant(q, K, N, ldq, scales, lds, group, zero, W, ldw, stream))


def gemm_int4_dequant_f32(q, K, N, ldq, scales, lds, group, zero, W, ldw, stream=0):
    _check(load().gemm_int4_dequant_f32(q, K, N, ldq, scales, lds, group, zero, W, ldw, stream))


def gemm_w4a16(M, N, K, alpha, X, ldx, qk, scales, lds, group, zero, beta, C, ldc, stream=0):
    _check(load().gemm_w4a16(M, N, K, alpha, X, ldx, qk, scales, lds, group, zero, beta, C, ldc,
                             stream))


def gemm_w4a16_f32out(M, N, K, alpha, X, ldx, qk, scales, lds, group, zero, beta, C, ldc, stream=0):
    _check(load().gemm_w4a16_f32out(M, N, K, alpha, X, ldx, qk, scales, lds, group, zero, beta, C, ldc,
                                    stream))


def gemm_w4_packed_bytes(K, N) -> int:
    return int(load().gemm_w4_packed_bytes(K, N))


def gemm_int4_repack(q, K, N, ldq, qk, stream=0):
    _check(load().gemm_int4_repack(q, K, N, ldq, qk, stream))


def gemm_attention(B, Hq, Hkv, Sq, Sk, D, Q, K, V, O, scale=0.0, causal=0, stream=0):
    _check(load().gemm_attention(B, Hq, Hkv, Sq, Sk, D, Q, K, V, O, scale, causal, stream))


def device_status(stream=0) -> tuple[int, int]:
    """(status code, location code) of the device status word; clears it."""
    where = ctypes.c_int(0)
    rc = load().gemm_device_status(stream, ctypes.byref(where))
    return rc, where.value


def force_path(path: int):
    _check(load().gemm_force_path(path))


def last_path() -> int:
    return load().gemm_last_path()


def force_tile_n(bn: int):
    _check(load().gemm_force_tile_n(bn))


def last_tile_n() -> int:
    return load().gemm_last_tile_n()


def force_tc_pair(mode: int):
    _check(load().gemm_force_tc_pair(mode))


def last_tc_pair() -> int:
    return load().gemm_last_tc_pair()


def force_split_tiles(enable: int):
    _check(load().gemm_force_split_tiles(enable))


def last_k_split() -> int:
    return load().gemm_last_k_split()


def set_wait_timeout_ns(ns: int):
    _check(load().gemm_set_wait_timeout_ns(ns))


def selftest_wait_timeout(ns: int, stream=0):
    _check(load().gemm_selftest_wait_timeout(ns, stream))


def test_stall(enable: int):
    """Test hook: later calls on this thread make one role of the first CTA
    wait on a barrier nothing arrives at, so the kernel's abort path runs."""
    _check(load().gemm_test_stall(int(enable)))

def _ld(t) -> int:
    """Leading dimension of a row-major 2-D tensor (unit stride along columns)."""
    if t.dim() != 2 or (t.stride(1) != 1 and t.shape[1] > 1):
        raise ValueError("expected a 2-D row-major tensor with unit column stride")
    return max(int(t.stride(0)), int(t.shape[1]), 1)


def gemm(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None, bias=None,
         act: int = ACT_NONE):
    """C = act(alpha*A@B + beta*C + bias) for CUDA tensors (fp32/fp32/fp32,
    bf16/bf16/bf16 or bf16/bf16/fp32; bias: N fp32 values or None).
    Argument marshalling only."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch {tuple(A.shape)} @ {tuple(B.shape)} -> {tuple(C.shape)}")
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("gemm() takes CUDA tensors")
    s = stream if stream is not None else torch.cuda.current_stream(A.device).cuda_stream
    args = (M, N, K, float(alpha), A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), float(beta),
            C.data_ptr(), _ld(C))
    if bias is not None:
        if bias.dtype != torch.float32 or not bias.is_cuda or bias.numel() != N or \
                (bias.dim() == 1 and bias.stride(0) != 1):
            raise ValueError("bias must be N contiguous fp32 values on the GPU")
    plain = bias is None and act == ACT_NONE
    ex = (bias.data_ptr() if bias is not None else None, int(act), s)
    if A.dtype == torch.float32 and B.dtype == torch.float32 and C.dtype == torch.float32:
        gemm_f32(*args, s) if plain else gemm_f32_ex(*args, *ex)
    elif A.dtype == torch.bfloat16 and B.dtype == torch.bfloat16 and C.dtype == torch.bfloat16:
        gemm_bf16(*args, s) if plain else gemm_bf16_ex(*args, *ex)
    elif A.dtype == torch.bfloat16 and B.dtype == torch.bfloat16 and C.dtype == torch.float32:
        gemm_bf16_f32out(*args, s) if plain else gemm_bf16_f32out_ex(*args, *ex)
    else:
        raise TypeError(f"unsupported dtypes {A.dtype}, {B.dtype} -> {C.dtype}")
    return C


def swiglu(A, Bgate, Bup, C, stream=None):
    """C = silu(A@Bgate) * (A@Bup) for bf16 CUDA tensors; Bgate and Bup share
    one shape and leading dimension.  Argument marshalling only."""
    import torch
    M, K = A.shape
    K2, N = Bgate.shape
    if K2 != K or tuple(Bup.shape) != (K, N) or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch {tuple(A.shape)} @ {tuple(Bgate.shape)}, "
                         f"{tuple(Bup.shape)} -> {tuple(C.shape)}")
    if _ld(Bgate) != _ld(Bup):
        raise ValueError("Bgate and Bup must have the same leading dimension")
    if not all(t.is_cuda and t.dtype == torch.bfloat16 for t in (A, Bgate, Bup, C)):
        raise TypeError("swiglu() takes bf16 CUDA tensors")
    s = stream if stream is not None else torch.cuda.current_stream(A.device).cuda_stream
    gemm_bf16_swiglu(M, N, K, A.data_ptr(), _ld(A), Bgate.data_ptr(), Bup.data_ptr(), _ld(Bgate),
                     C.data_ptr(), _ld(C), s)
    return C


def gemm_fp8_tensors(A, fmt_a: int, B, fmt_b: int, C, alpha: float = 1.0, beta: float = 0.0,
                     stream=None):
    """C = alpha*dec(A)@dec(B) + beta*C for CUDA tensors of FP8 codes (uint8)
    and a bf16 or fp32 C.  Argument marshalling only."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch {tuple(A.shape)} @ {tuple(B.shape)} -> {tuple(C.shape)}")
    if A.dtype != torch.uint8 or B.dtype != torch.uint8 or not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise TypeError("gemm_fp8_tensors() takes uint8 FP8 codes on the GPU")
    s = stream if stream is not None else torch.cuda.current_stream(A.device).cuda_stream
    args = (M, N, K, float(alpha), A.data_ptr(), int(fmt_a), _ld(A), B.data_ptr(), int(fmt_b), _ld(B),
            float(beta), C.data_ptr(), _ld(C), s)
    if C.dtype == torch.bfloat16:
        gemm_fp8(*args)
    elif C.dtype == torch.float32:
        gemm_fp8_f32out(*args)
    else:
        raise TypeError(f"unsupported output dtype {C.dtype}")
    return C


def int4_dequant(q, scales, N: int, group: int, zero: int, W, stream=None):
    """W = scales[k // group][n] * (q[k][n] - zero) for CUDA tensors: q K x ceil(N/2)
    uint8 codes, scales bf16, W bf16 or fp32 (K x N).  Argument marshalling only."""
    import torch
    K = q.shape[0]
    if W.shape[0] != K or W.shape[1] != N or q.dtype != torch.uint8 or scales.dtype != torch.bfloat16:
        raise ValueError("int4_dequant(): shape or dtype mismatch")
    s = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    args = (q.data_ptr(), K, N, _ld(q), scales.data_ptr(), _ld(scales), group, zero, W.data_ptr(),
            _ld(W), s)
    if W.dtype == torch.bfloat16:
        gemm_int4_dequant(*args)
    elif W.dtype == torch.float32:
        gemm_int4_dequant_f32(*args)
    else:
        raise TypeError(f"unsupported output dtype {W.dtype}")
    return W



def int4_repack(q, K: int, N: int, stream=None):
    """Tiled copy (a new flat CUDA uint8 tensor of gemm_w4_packed_bytes(K, N))
    of INT4 codes q (K x ceil(N/2) bytes, packed along n).  Argument
    marshalling only."""
    import torch
    qk = torch.empty((max(gemm_w4_packed_bytes(K, N), 16),), dtype=torch.uint8, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    gemm_int4_repack(q.data_ptr(), K, N, _ld(q), qk.data_ptr(), s)
    return qk


def w4a16(X, qk, scales, group: int, zero: int, C, alpha: float = 1.0, beta: float = 0.0,
          stream=None):
    """C = alpha * X @ W + beta * C with W = scales[k // group] * (q - zero) given
    as K-packed codes qk (from int4_repack); X bf16, C bf16 or fp32.  Argument
    marshalling only."""
    import torch
    M, K = X.shape
    N = C.shape[1]
    if C.shape[0] != M or qk.numel() < gemm_w4_packed_bytes(K, N) or X.dtype != torch.bfloat16:
        raise ValueError("w4a16(): shape or dtype mismatch")
    s = stream if stream is not None else torch.cuda.current_stream(X.device).cuda_stream
    args = (M, N, K, float(alpha), X.data_ptr(), _ld(X), qk.data_ptr(), scales.data_ptr(),
            _ld(scales), int(group), int(zero), float(beta), C.data_ptr(), _ld(C), s)
    if C.dtype == torch.bfloat16:
        gemm_w4a16(*args)
    elif C.dtype == torch.float32:
        gemm_w4a16_f32out(*args)
    else:
        raise TypeError(f"unsupported output dtype {C.dtype}")
    return C


def attention(Q, K, V, O, scale: float = 0.0, causal: bool = False, stream=None):
    """O = softmax(Q K^T * scale) V for contiguous bf16 CUDA tensors Q, O
    [B][Hq][Sq][D] and K, V [B][Hkv][Sk][D] (scale 0: 1/sqrt(D)).  Argument
    marshalling only."""
    import torch
    B, Hq, Sq, D = Q.shape
    Hkv, Sk = K.shape[1], K.shape[2]
    for t in (Q, K, V, O):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise TypeError("attention() takes contiguous bf16 CUDA tensors")
    if tuple(V.shape) != tuple(K.shape) or tuple(O.shape) != tuple(Q.shape) or K.shape[0] != B or K.shape[3] != D:
        raise ValueError("attention(): shape mismatch")
    s = stream if stream is not None else torch.cuda.current_stream(Q.device).cuda_stream
    gemm_attention(B, Hq, Hkv, Sq, Sk, D, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                   float(scale), int(bool(causal)), s)
    return O
