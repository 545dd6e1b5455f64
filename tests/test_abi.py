"""The C-ABI library builds, loads without a GPU, and exports every declared symbol."""
import ctypes
import glob
import os
import re
import shutil
import subprocess

import pytest

from conftest import ROOT

HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def _declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h, encoding="utf-8").read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(gemm_\w+)\s*\(", src,
                                flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib_path():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from roofline_driven_optimisation_gb300 import _build
    return _build.build()


def test_header_declares_the_abi():
    names = _declared_functions()
    for want in ("gemm_f32", "gemm_bf16", "gemm_bf16_f32out", "gemm_get_last_error",
                 "gemm_device_status", "gemm_bf16_swiglu", "gemm_test_stall"):
        assert want in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    import roofline_driven_optimisation_gb300 as g
    assert sorted(g.EXPORTS) == _declared_functions()


def test_library_exports_no_torch_symbols(lib_path):
    r = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm unavailable")
    exported = [ln.split()[-1] for ln in r.stdout.splitlines() if " T " in ln]
    gemm_syms = [s for s in exported if s.startswith("gemm_")]
    assert sorted(gemm_syms) == _declared_functions()
    assert not any("torch" in s or "at::" in s for s in exported)


def test_header_is_valid_c(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc unavailable")
    src = tmp_path / "use.c"
    src.write_text('#include "gb300gemm.h"\n'
                   'int main(void){ return gemm_get_last_error() == 0; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include", str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_calls_fail_cleanly_without_gpu(lib_path):
    import torch
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    import roofline_driven_optimisation_gb300 as g
    g.load()
    # argument validation happens before any device access
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32(-1, 4, 4, 1.0, 0, 4, 0, 4, 0.0, 0, 4, 0)
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_bf16(4, 4, 8, 1.0, 16, 4, 16, 4, 0.0, 16, 4, 0)   # lda < K
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_bf16(4, 4, 4, 1.0, 17, 4, 32, 4, 0.0, 64, 4, 0)   # odd address for bf16
    assert e.value.code == g.GEMM_ERR_MISALIGNED
    # M == 0 is a no-op that touches nothing
    g.gemm_f32(0, 4, 4, 1.0, 0, 4, 0, 4, 0.0, 0, 4, 0)
    # a real call needs a device: it must report an error, never compute on the CPU
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32(4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, 0)
    assert e.value.code in (g.GEMM_ERR_CUDA, g.GEMM_ERR_UNSUPPORTED)


def test_force_path_validation(lib_path):
    import roofline_driven_optimisation_gb300 as g
    g.load()
    with pytest.raises(g.GemmError):
        g.force_path(99)
    g.force_path(g.PATH_AUTO)
