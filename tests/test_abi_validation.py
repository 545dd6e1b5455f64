"""Argument validation of every C-ABI entry point, on the CPU: each bad call
returns its gemm_status and a message before any device access, and calls of
size zero are no-ops that touch nothing.  (Without a GPU every call that
passes validation fails with GEMM_ERR_CUDA or GEMM_ERR_UNSUPPORTED; the GPU
tests cover the rest.)"""
import shutil
import os

import pytest


@pytest.fixture(scope="module")
def g():
    import torch
    if torch.cuda.is_available():
        pytest.skip("runs only where validation is all that can happen")
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from roofline_driven_optimisation_gb300 import _build
    _build.build()
    import roofline_driven_optimisation_gb300 as lib
    lib.load()
    return lib


P = 1 << 20          # an aligned stand-in address (never dereferenced)
S = 0                # default stream

CASES = [
    # (entry point, args, status name, message fragment)
    ("gemm_f32", (4, -1, 4, 1.0, P, 4, P, 4, 0.0, P, 4, S), "GEMM_ERR_INVALID_ARG", "negative size"),
    ("gemm_f32", (4, 4, 4, 1.0, P, 4, P, 3, 0.0, P, 4, S), "GEMM_ERR_INVALID_ARG", "leading dimension"),
    ("gemm_f32", (4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 3, S), "GEMM_ERR_INVALID_ARG", "leading dimension"),
    ("gemm_f32", (4, 4, 4, 1.0, P, 4, P, 4, 0.0, 0, 4, S), "GEMM_ERR_INVALID_ARG", "C is NULL"),
    ("gemm_f32", (4, 4, 4, 1.0, 0, 4, P, 4, 0.0, P, 4, S), "GEMM_ERR_INVALID_ARG", "A or B is NULL"),
    ("gemm_f32", (4, 4, 4, 1.0, P + 2, 4, P, 4, 0.0, P, 4, S), "GEMM_ERR_MISALIGNED", "not aligned"),
    ("gemm_bf16_f32out", (4, 4, 4, 1.0, P, 4, P, 4, 0.0, P + 2, 4, S), "GEMM_ERR_MISALIGNED",
     "not aligned"),
    ("gemm_f32_ex", (4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, 0, 7, S), "GEMM_ERR_INVALID_ARG",
     "unknown activation"),
    ("gemm_f32_ex", (4, 4, 4, 1.0, P, 4, P, 4, 0.0, P, 4, P + 2, 1, S), "GEMM_ERR_MISALIGNED",
     "bias"),
    ("gemm_bf16_swiglu", (4, 4, 4, P, 4, P, 0, 4, P, 4, S), "GEMM_ERR_INVALID_ARG", "NULL"),
    ("gemm_fp8", (4, 4, 4, 1.0, P, 2, 4, P, 0, 4, 0.0, P, 4, S), "GEMM_ERR_INVALID_ARG",
     "FP8 format"),
    ("gemm_int4_dequant", (P, 64, 8, 4, P, 8, 0, 8, P, 8, S), "GEMM_ERR_INVALID_ARG", "group size"),
    ("gemm_int4_dequant", (P, 64, 8, 4, P, 8, 32, 16, P, 8, S), "GEMM_ERR_INVALID_ARG", "zero point"),
    ("gemm_int4_dequant", (P, 64, 8, 3, P, 8, 32, 8, P, 8, S), "GEMM_ERR_INVALID_ARG",
     "leading dimension"),
    ("gemm_int4_repack", (P, 64, 8, 4, P + 8, S), "GEMM_ERR_MISALIGNED", "16-byte"),
    ("gemm_w4a16", (4, 8, 64, 1.0, P, 64, P, P, 8, 128, -1, 1.0, P, 8, S), "GEMM_ERR_INVALID_ARG",
     "zero point"),
    ("gemm_w4a16", (4, 8, 64, 1.0, P, 64, P + 4, P, 8, 128, 8, 1.0, P, 8, S), "GEMM_ERR_MISALIGNED",
     "16-byte"),
    ("gemm_w4a16", (4, 8, 64, 1.0, P, 64, P, P, 8, 128, 8, 1.0, 0, 8, S), "GEMM_ERR_INVALID_ARG",
     "C is NULL"),
    ("gemm_attention", (1, 6, 4, 16, 16, 64, P, P, P, P, 0.0, 0, S), "GEMM_ERR_INVALID_ARG",
     "multiple of Hkv"),
    ("gemm_attention", (1, 4, 4, 16, 16, 0, P, P, P, P, 0.0, 0, S), "GEMM_ERR_INVALID_ARG", "bad sizes"),
    ("gemm_attention", (1, 4, 4, 16, 16, 64, P, P, P, P, -1.0, 0, S), "GEMM_ERR_INVALID_ARG",
     "bad scale"),
    ("gemm_attention", (1, 4, 4, 16, 16, 64, P + 1, P, P, P, 0.0, 0, S), "GEMM_ERR_MISALIGNED",
     "aligned"),
    ("gemm_attention", (2048, 64, 8, 16, 16, 64, P, P, P, P, 0.0, 0, S), "GEMM_ERR_UNSUPPORTED",
     "exceeds 65535"),
]


@pytest.mark.parametrize("fn,args,status,fragment", CASES)
def test_bad_arguments_are_rejected(g, fn, args, status, fragment):
    with pytest.raises(g.GemmError) as e:
        getattr(g, fn)(*args)
    assert e.value.code == getattr(g, status), str(e.value)
    assert fragment in str(e.value), str(e.value)


NO_OPS = [
    ("gemm_f32", (0, 4, 4, 1.0, 0, 4, 0, 4, 0.0, 0, 4, S)),
    ("gemm_bf16", (4, 0, 4, 1.0, 0, 4, 0, 1, 0.0, 0, 1, S)),
    ("gemm_int4_dequant", (0, 0, 8, 4, 0, 8, 32, 8, 0, 8, S)),
    ("gemm_int4_repack", (0, 64, 0, 1, 0, S)),
    ("gemm_w4a16", (0, 8, 64, 1.0, 0, 64, 0, 0, 8, 128, 8, 1.0, 0, 8, S)),
    ("gemm_attention", (0, 4, 4, 16, 16, 64, 0, 0, 0, 0, 0.0, 1, S)),
]


@pytest.mark.parametrize("fn,args", NO_OPS)
def test_empty_calls_are_no_ops(g, fn, args):
    getattr(g, fn)(*args)   # no GPU here: any device access would raise


def test_wait_limit_is_clamped(g):
    # 1 ms .. 10 s, 0 restores the default; outside the range is refused and
    # leaves the limit as it was
    for bad in (1, 999_999, 10_000_000_001, (1 << 64) - 1):
        with pytest.raises(g.GemmError) as e:
            g.set_wait_timeout_ns(bad)
        assert e.value.code == g.GEMM_ERR_INVALID_ARG
        assert "outside" in str(e.value)
    for ok in (1_000_000, 2_500_000, 10_000_000_000, 0):
        g.set_wait_timeout_ns(ok)


def test_stall_hook_validation(g):
    for bad in (-1, 2):
        with pytest.raises(g.GemmError) as e:
            g.test_stall(bad)
        assert e.value.code == g.GEMM_ERR_INVALID_ARG
    g.test_stall(1)
    g.test_stall(0)
