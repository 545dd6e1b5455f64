"""Measurement probes used by bench.py and the GPU tests, built as their own
shared library (libgb300probe.so) so that the GEMM library holds only the
GEMM path.

probe_fp32_fma: an FP32 FMA throughput kernel that checks the FP32 roofline's
peak (SMs x 128 lanes x 2 FLOP x SM clock) on the device, with scalar and with
packed f32x2 FMAs.
probe_read_stream, probe_empty: the floors of a kernel timed alone between two
events -- a read-only pass over the same bytes, and an empty launch.
probe_hold: keeps the stream busy for a while, so that a batch of timed
launches enqueued meanwhile never waits for the host.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgb300probe.so")
SOURCES = [os.path.join(HERE, "fma_probe.cu")]
DEPS = SOURCES + [os.path.join(HERE, "gb300probe.h"), os.path.abspath(__file__)]

_lib = None
_lock = threading.Lock()


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False) -> str:
    """Compile the probe library for sm_103a (in-tree, one nvcc call)."""
    if not force and up_to_date():
        return LIB_PATH
    from roofline_driven_optimisation_gb300 import _build
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [_build.nvcc()] + _build.ARCH_FLAGS + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                                                 "-I", HERE, "-shared", "-o", tmp] + SOURCES
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on the probe library:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run bench_probe.build()")
        lib = ctypes.CDLL(LIB_PATH)
        i, vp = ctypes.c_int, ctypes.c_void_p
        lib.probe_fp32_fma.argtypes = [i, i, vp, ctypes.POINTER(ctypes.c_double), vp]
        lib.probe_fp32_fma.restype = i
        lib.probe_read_stream.argtypes = [vp, ctypes.c_size_t, vp, vp]
        lib.probe_read_stream.restype = i
        lib.probe_empty.argtypes = [vp]
        lib.probe_empty.restype = i
        lib.probe_hold.argtypes = [ctypes.c_ulonglong, vp]
        lib.probe_hold.restype = i
        _lib = lib
        return lib


def probe_fp32_fma(packed: bool, iters: int, sink_ptr: int, stream=0) -> float:
    """Launch the FP32 FMA throughput probe; returns the launch's FLOPs.
    Raises ValueError for bad arguments and RuntimeError if a CUDA call failed."""
    flops = ctypes.c_double(0.0)
    rc = load().probe_fp32_fma(int(bool(packed)), int(iters), sink_ptr, ctypes.byref(flops), stream)
    if rc == 1:
        raise ValueError("probe_fp32_fma: iters <= 0 or a NULL pointer")
    if rc != 0:
        raise RuntimeError(f"probe_fp32_fma: launch failed ({rc})")
    return flops.value


def probe_read_stream(buf_ptr: int, nbytes: int, sink_ptr: int, stream=0):
    """Launch a read-only streaming pass over nbytes of device memory."""
    rc = load().probe_read_stream(buf_ptr, int(nbytes), sink_ptr, stream)
    if rc == 1:
        raise ValueError("probe_read_stream: NULL, unaligned or ragged buffer")
    if rc != 0:
        raise RuntimeError(f"probe_read_stream: launch failed ({rc})")


def probe_empty(stream=0):
    """Launch one empty CTA."""
    if load().probe_empty(stream) != 0:
        raise RuntimeError("probe_empty: launch failed")


def probe_hold(ns: int, stream=0):
    """Keep `stream` busy for ns nanoseconds (<= 1e9) of device time."""
    rc = load().probe_hold(int(ns), stream)
    if rc != 0:
        raise RuntimeError(f"probe_hold failed ({rc})")
