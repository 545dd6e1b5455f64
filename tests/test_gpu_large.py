"""GEMMs with one operand past 2^31 elements, checked on sampled rows and
columns against the fp64 oracle with the plain max sum_k |A||B| scale.

Every element offset in the kernels is 64-bit while tile counts and TMA
coordinates stay small, so an offset computed in 32 bits anywhere would show
here as wrong or missing values in the last rows or columns.  Only the
sampled rows and columns of C come back to the host."""
import numpy as np
import pytest
import torch

import oracle
import roofline_driven_optimisation_gb300 as g
from roofline_driven_optimisation_gb300 import inputs

pytestmark = pytest.mark.gpu


def _status_ok():
    torch.cuda.synchronize()
    status, where = g.device_status()
    assert status == 0, f"device status {status} at site {where}"


def _samples(n, extra, seed):
    rng = np.random.default_rng(seed)
    picks = rng.choice(n, 12, replace=False)
    return sorted(set(int(x) for x in picks) | {0, n - 1} | set(extra))


def _check(A_cpu, B_rows_cpu, B_cols_cpu, C_rows, C_cols, rows, cols, alpha, tol):
    """A_cpu: all of A; B_rows_cpu: all of B (or None when B stays on the
    device); B_cols_cpu: B[:, cols]; C_rows / C_cols: the GPU's C[rows] and
    C[:, cols]."""
    worst = 0.0
    parts = [(A_cpu, B_cols_cpu, C_cols)]
    if B_rows_cpu is not None:
        parts.append((A_cpu[rows], B_rows_cpu, C_rows))
    for A_s, B_s, got in parts:
        ref = oracle.gemm(A_s, B_s, alpha, 0.0, None)
        plain = oracle.abs_product_max(A_s, B_s)
        worst = max(worst, oracle.normwise_error(got, ref, plain * abs(alpha)))
    assert worst <= tol, f"sampled normwise error {worst:.3e} > {tol:g}"


def test_bf16_pairs_c_past_2_31_elements(cuda_lib):
    # 65536 x 40000 bf16 C (2.62e9 elements): rows from 53688 on start past 2^31
    M, N, K = 65536, 40000, 64
    A = inputs.random_matrix(M, K, seed=61, dtype="bf16")
    B = inputs.random_matrix(K, N, seed=62, dtype="bf16")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.gemm(A.cuda(), B.cuda(), C)
    assert g.last_path() == g.PATH_BF16_TC
    _status_ok()
    rows = _samples(M, [53687, 53688], 1)
    cols = _samples(N, [], 2)
    C_rows, C_cols = C[rows].cpu(), C[:, cols].cpu()
    del C
    _check(A, B, B[:, cols], C_rows, C_cols, rows, cols, 1.0, oracle.TOL_BF16_OUT)


def test_fp32_simt_c_past_2_31_elements(cuda_lib):
    # 65536 x 33024 fp32 C (2.16e9 elements, 8.7 GB), alpha 1.5
    M, N, K = 65536, 33024, 32
    A = inputs.random_matrix(M, K, seed=63)
    B = inputs.random_matrix(K, N, seed=64)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g.gemm(A.cuda(), B.cuda(), C, 1.5)
    assert g.last_path() == g.PATH_F32_SIMT
    _status_ok()
    rows = _samples(M, [65028, 65029], 3)
    cols = _samples(N, [], 4)
    C_rows, C_cols = C[rows].cpu(), C[:, cols].cpu()
    del C
    _check(A, B, B[:, cols], C_rows, C_cols, rows, cols, 1.5, oracle.TOL_F32)


def test_decode_weight_past_2_31_elements(cuda_lib):
    # M = 4 against a 65536 x 36864 bf16 weight (2.42e9 elements, 4.8 GB),
    # drawn on the device; every column's last 7000 rows lie past 2^31
    M, N, K = 4, 36864, 65536
    A = inputs.random_matrix(M, K, seed=65, dtype="bf16")
    B = inputs.device_uniform(K, N, seed=66, device="cuda", dtype="bf16")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.gemm(A.cuda(), B, C)
    assert g.last_path() == g.PATH_SKINNY
    _status_ok()
    cols = _samples(N, [], 5)
    B_cols = B[:, cols].cpu()
    C_cols = C[:, cols].cpu()
    del B, C
    _check(A, None, B_cols, None, C_cols, list(range(M)), cols, 1.0, oracle.TOL_BF16_OUT)


def test_fp8_pairs_c_past_2_31_elements(cuda_lib):
    # 65536 x 40000 bf16 C from E4M3 codes (K = 128: one stage)
    from oracle import fp8
    M, N, K = 65536, 40000, 128
    c = inputs.make_fp8(M, N, K, inputs.FP8_E4M3, inputs.FP8_E4M3, seed=67)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.gemm_fp8_tensors(c.A.cuda(), c.fmt_a, c.B.cuda(), c.fmt_b, C, c.alpha)
    assert g.last_path() == g.PATH_BF16_TC
    _status_ok()
    rows = _samples(M, [53687, 53688], 6)
    cols = _samples(N, [], 7)
    C_rows, C_cols = C[rows].cpu(), C[:, cols].cpu()
    del C
    worst = 0.0
    for A_s, B_s, got in ((c.A[rows], c.B, C_rows), (c.A, c.B[:, cols], C_cols)):
        ref = fp8.gemm_fp8(A_s, c.fmt_a, B_s, c.fmt_b, c.alpha)
        den = fp8.normwise_denominator_fp8(A_s, c.fmt_a, B_s, c.fmt_b, c.alpha)
        worst = max(worst, oracle.normwise_error(got, ref, den))
    assert worst <= oracle.TOL_BF16_OUT, worst
