"""Fused FFN gate/up pair, C = silu(A*Bgate) * (A*Bup), through the C ABI on
every kernel family (decode kernel, CTA pairs, generic), against the fp64
oracle.  The error scale is oracle.epilogue.swiglu_error_scale: the
first-order sensitivity of silu(g)*u to errors in g and u of the size of
sum_k |A||B|, which also bounds the final rounding to bf16."""
import numpy as np
import pytest
import torch

import oracle
import roofline_driven_optimisation_gb300 as g
from oracle import epilogue as E
from roofline_driven_optimisation_gb300 import inputs

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16
TOL = oracle.TOL_BF16_OUT


def _place(x, pad, off, fill=0.0):
    """x (CPU) copied into a device buffer with `pad` extra columns per row
    and the matrix starting `off` elements past an aligned base."""
    rows, cols = x.shape
    ld = max(cols + pad, 1)
    flat = torch.full((off + rows * ld + 8,), fill, dtype=x.dtype)
    flat[off:off + rows * ld].view(rows, ld)[:, :cols] = x
    d = flat.cuda()
    return d, d.data_ptr() + off * d.element_size(), ld


def _run(c, *, pad=(0, 0, 0), offset=(0, 0, 0), path=None):
    M, K = c.A.shape
    N = c.Bgate.shape[1]
    A_d, a_ptr, lda = _place(c.A, pad[0], offset[0])
    Bg_d, bg_ptr, ldb = _place(c.Bgate, pad[1], offset[1])
    Bu_d, bu_ptr, _ = _place(c.Bup, pad[1], offset[1])
    C_d, c_ptr, ldc = _place(torch.full((M, N), float("nan"), dtype=BF16), pad[2], offset[2],
                             fill=float("nan"))
    if path is not None:
        g.force_path(path)
    try:
        g.gemm_bf16_swiglu(M, N, K, a_ptr, lda, bg_ptr, bu_ptr, ldb, c_ptr, ldc,
                           torch.cuda.current_stream().cuda_stream)
        ran = g.last_path()
    finally:
        g.force_path(g.PATH_AUTO)
    torch.cuda.synchronize()
    status, where = g.device_status()
    assert status == 0, f"device status {status} at site {where}"
    full = C_d.cpu()[offset[2]:offset[2] + M * ldc].view(M, ldc)
    if pad[2]:
        assert torch.isnan(full[:, N:].float()).all(), "row padding of C was written"
    return full[:, :N].clone(), ran


def _check(c, **kw):
    C, ran = _run(c, **kw)
    ref = E.swiglu(c.A, c.Bgate, c.Bup)
    scale = E.swiglu_error_scale(c.A, c.Bgate, c.Bup)
    err = oracle.normwise_error(C, ref, scale if scale else 1.0)
    assert err <= TOL, f"normwise error {err:.3e} > {TOL:g} (path {g.PATH_NAMES.get(ran)})"
    return err, ran


def _expected_split(N, K):
    """K split of the decode kernel: the largest power of two <= 8 that keeps
    the grid (64-column tiles x split) within two CTAs per SM, and no more
    than the K stages of 64."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles_n, k_tiles = -(-N // 64), -(-K // 64)
    s = 1
    while s * 2 <= 8 and tiles_n * s * 2 <= 2 * sms:
        s *= 2
    while s > 1 and s > k_tiles:
        s //= 2
    return s


# LLaMA-7B FFN gate/up (K = 4096, N = 11008) at the decode batch sizes
@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_llama_gate_up(cuda_lib, M):
    _, ran = _check(inputs.make_swiglu(M))
    assert ran == g.PATH_SKINNY
    assert g.last_k_split() == _expected_split(11008, 4096)


# tiles of 64 output columns: N = 4096 gives a K split of 4, N = 200 a ragged
# last tile and (K = 136: three K stages) a split capped at 2
@pytest.mark.parametrize("M,N,K", [(3, 4096, 1024), (16, 200, 136), (7, 64, 64), (2, 8, 4096)])
def test_decode_splits_and_tails(cuda_lib, M, N, K):
    _, ran = _check(inputs.make_swiglu(M, N, K, seed=M + N))
    assert ran == g.PATH_SKINNY
    assert g.last_k_split() == _expected_split(N, K)


@pytest.mark.parametrize("M,N,K", [(300, 520, 256), (17, 128, 64), (256, 11008, 64),
                                   (512, 1000, 1000)])
def test_cta_pair_tiles(cuda_lib, M, N, K):
    _, ran = _check(inputs.make_swiglu(M, N, K, seed=M))
    assert ran == g.PATH_BF16_TC
    assert g.last_tc_pair() == 2 and g.last_tile_n() == 128


def test_prefill_llama_gate_up_sampled(cuda_lib):
    # M = 2048 tokens through the LLaMA-7B gate/up pair (the size the pair
    # kernel is timed at), checked on sampled rows and columns
    c = inputs.make_swiglu(2048)
    C, ran = _run(c)
    assert ran == g.PATH_BF16_TC
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(2048, 12, replace=False))
    rows[-1] = 2047
    cols = np.sort(rng.choice(11008, 40, replace=False))
    cols[-1] = 11007
    worst = 0.0
    for A_s, Bg_s, Bu_s, got in ((c.A[rows], c.Bgate, c.Bup, C[rows]),
                                 (c.A, c.Bgate[:, cols], c.Bup[:, cols], C[:, cols])):
        ref = E.swiglu(A_s, Bg_s, Bu_s)
        scale = E.swiglu_error_scale(A_s, Bg_s, Bu_s)
        worst = max(worst, oracle.normwise_error(got, ref, scale))
    assert worst <= TOL, f"sampled normwise error {worst:.3e}"


@pytest.mark.parametrize("M", [5, 40])
def test_generic_kernel(cuda_lib, M):
    c = inputs.make_swiglu(M, 90, 70, seed=9)   # odd sizes: no TMA path
    _, ran = _check(c)
    assert ran == g.PATH_GENERIC
    _, ran = _check(inputs.make_swiglu(M, 128, 64, seed=9), path=g.PATH_GENERIC)
    assert ran == g.PATH_GENERIC


def test_padded_leading_dimensions(cuda_lib):
    # padded leading dimensions that stay multiples of 16 bytes: fast paths
    _, ran = _check(inputs.make_swiglu(9, 300, 200, seed=2), pad=(8, 20, 8))
    assert ran == g.PATH_SKINNY
    _, ran = _check(inputs.make_swiglu(130, 300, 200, seed=2), pad=(8, 20, 8))
    assert ran == g.PATH_BF16_TC
    # an element offset breaks 16-byte alignment: the generic kernel
    _, ran = _check(inputs.make_swiglu(130, 300, 200, seed=2), offset=(1, 3, 1))
    assert ran == g.PATH_GENERIC


def test_forced_paths_agree(cuda_lib):
    c = inputs.make_swiglu(16, 256, 512, seed=4)
    for path in (g.PATH_SKINNY, g.PATH_BF16_TC, g.PATH_GENERIC):
        C, ran = _run(c, path=path)
        assert ran == path
        ref = E.swiglu(c.A, c.Bgate, c.Bup)
        assert oracle.normwise_error(C, ref, E.swiglu_error_scale(c.A, c.Bgate, c.Bup)) <= TOL
    with pytest.raises(g.GemmError) as e:
        g.force_path(g.PATH_F32_SIMT)
        try:
            _run(c)
        finally:
            g.force_path(g.PATH_AUTO)
    assert e.value.code == g.GEMM_ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [4, 300])
def test_deterministic(cuda_lib, M):
    c = inputs.make_swiglu(M, 1024, 2048, seed=6)
    C1, _ = _run(c)
    C2, _ = _run(c)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


def test_k_zero_and_arguments(cuda_lib):
    M, N = 5, 40
    C = torch.full((M, N), float("nan"), dtype=BF16, device="cuda")
    A = torch.zeros((M, 1), dtype=BF16, device="cuda")
    Bg = torch.zeros((1, N), dtype=BF16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # K == 0: silu(0) * 0 = 0, and neither weight is read (Bup may be NULL)
    g.gemm_bf16_swiglu(M, N, 0, A.data_ptr(), 1, Bg.data_ptr(), None, N, C.data_ptr(), N, s)
    torch.cuda.synchronize()
    assert torch.equal(C.float().cpu(), torch.zeros((M, N)))
    with pytest.raises(g.GemmError) as e:
        g.gemm_bf16_swiglu(M, N, 1, A.data_ptr(), 1, Bg.data_ptr(), None, N, C.data_ptr(), N, s)
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_bf16_swiglu(M, N, 1, A.data_ptr(), 1, Bg.data_ptr(), Bg.data_ptr() + 1, N,
                           C.data_ptr(), N, s)
    assert e.value.code == g.GEMM_ERR_MISALIGNED
    # M == 0 or N == 0: nothing runs
    g.gemm_bf16_swiglu(0, N, 1, None, 1, None, None, N, None, N, s)


def test_tensor_binding(cuda_lib):
    c = inputs.make_swiglu(24, 256, 128, seed=8)
    out = torch.empty((24, 256), dtype=BF16, device="cuda")
    g.swiglu(c.A.cuda(), c.Bgate.cuda(), c.Bup.cuda(), out)
    torch.cuda.synchronize()
    ref = E.swiglu(c.A, c.Bgate, c.Bup)
    assert oracle.normwise_error(out.cpu(), ref, E.swiglu_error_scale(c.A, c.Bgate, c.Bup)) <= TOL
    with pytest.raises(ValueError):
        g.swiglu(c.A.cuda(), c.Bgate.cuda(), c.Bup[:, :128].cuda(), out)
