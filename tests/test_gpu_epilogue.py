"""Fused epilogue C = act(alpha*A*B + beta*C + bias) on every kernel family,
against the fp64 oracle.  The error scale is that of the pre-activation value
(|alpha| sum|A||B| + |beta||C0| + |bias|); the activations' slopes are <= 1.13."""
import pytest
import torch

import oracle
import roofline_driven_optimisation_gb300 as g
from oracle import epilogue as E
from roofline_driven_optimisation_gb300 import inputs

pytestmark = pytest.mark.gpu
F32, BF16 = torch.float32, torch.bfloat16
ACTS = [g.ACT_NONE, g.ACT_RELU, g.ACT_SILU, g.ACT_GELU]


def _run(case, out, alpha, beta, with_bias, act, *, path=None, pair=None, bn=None):
    A, B = case.A.cuda(), case.B.cuda()
    M, N = case.A.shape[0], case.B.shape[1]
    C0 = case.C0.to(out) if (beta != 0 and case.C0 is not None) else None
    C = C0.cuda() if C0 is not None else torch.full((M, N), float("nan"), dtype=out, device="cuda")
    bias = inputs.random_matrix(1, N, 77, dist="normal").reshape(N) if with_bias else None
    for fn, v in ((g.force_path, path), (g.force_tc_pair, pair), (g.force_tile_n, bn)):
        if v is not None:
            fn(v)
    try:
        g.gemm(A, B, C, alpha, beta, bias=bias.cuda() if bias is not None else None, act=act)
        torch.cuda.synchronize()
        ran = g.last_path()
    finally:
        g.force_path(g.PATH_AUTO)
        g.force_tc_pair(0)
        g.force_tile_n(0)
    assert g.device_status()[0] == 0
    ref = E.gemm_epilogue(case.A, case.B, alpha, beta, C0, bias, act)
    denom = oracle.normwise_denominator(case.A, case.B, alpha, beta, C0, bias=bias)
    err = oracle.normwise_error(C.cpu(), ref, denom)
    tol = {F32: oracle.TOL_F32 if case.A.dtype == F32 else oracle.TOL_BF16_F32OUT,
           BF16: oracle.TOL_BF16_OUT}[out]
    assert err <= tol, f"act {act} bias {with_bias}: err {err:.3e} > {tol:g} (path {ran})"
    return ran


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("with_bias", [False, True])
def test_fp32_simt_and_generic(cuda_lib, act, with_bias):
    c = inputs.make("fp32_4096", M=200, N=264, K=128)
    assert _run(c, F32, 1.5, 0.5, with_bias, act) == g.PATH_F32_SIMT
    for bn in (128, 256):   # both register tiles
        assert _run(c, F32, 1.5, 0.5, with_bias, act, bn=bn) == g.PATH_F32_SIMT
    assert _run(c, F32, 1.0, 0.0, with_bias, act, path=g.PATH_GENERIC) == g.PATH_GENERIC
    c2 = inputs.make("fp32_4096", M=70, N=90, K=52)   # N not a multiple of 4: scalar tail
    _run(c2, F32, 1.5, 0.5, with_bias, act)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("bn", [128, 256])
def test_fp32_split_last_wave(cuda_lib, act, bn):
    # nine (six) tiles with K = 1024: each tile's K range is split over four
    # CTAs of a cluster (or stream-K over 24 CTAs), and the CTA that sums a
    # block applies beta, bias and activation
    c = inputs.make("fp32_4096", M=300, N=264, K=1024)
    assert _run(c, F32, 1.5, 0.5, True, act, bn=bn) == g.PATH_F32_SIMT
    assert g.last_k_split() == 4 if bn == 128 else g.last_k_split() >= 2
    _run(c, F32, 1.0, 0.0, False, act, bn=bn)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("out", [BF16, F32])
@pytest.mark.parametrize("sched", [(1, 256), (1, 128), (2, 256), (2, 128)])
def test_bf16_tensor_core(cuda_lib, act, out, sched):
    pair, bn = sched
    c = inputs.make("decode_m16_o", M=300, N=520, K=256)
    assert _run(c, out, 1.0, 1.0, True, act, pair=pair, bn=bn) == g.PATH_BF16_TC
    assert g.last_tile_n() == bn


@pytest.mark.parametrize("act", [g.ACT_SILU, g.ACT_GELU])
def test_bf16_pair_half_width_schedule(cuda_lib, act):
    c = inputs.make("decode_m16_o", M=1536, N=1280, K=256)
    _run(c, BF16, 1.0, 1.0, True, act, pair=2, bn=256)
    assert g.last_tc_pair() == 4


@pytest.mark.parametrize("act", [g.ACT_RELU, g.ACT_GELU])
@pytest.mark.parametrize("out", [BF16, F32])
def test_bf16_pair_stream_k_schedule(cuda_lib, act, out):
    # the finisher of a stream-K tile applies beta, bias and the activation
    # once, after the partial tiles are added
    c = inputs.make("decode_m16_o", M=1536, N=1280, K=1024)
    g.force_split_tiles(2)
    try:
        _run(c, out, 1.5, 0.5, True, act, pair=2, bn=256)
        assert g.last_tc_pair() == 6
    finally:
        g.force_split_tiles(1)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("m,N", [(4, 512), (16, 520), (1, 20480), (16, 20480)])
def test_skinny(cuda_lib, act, m, N):
    # N = 20480: 160 column tiles, split 1 (direct epilogue); N = 512: split-K
    c = inputs.make(f"decode_m{m}_o", M=m, N=N, K=256)
    for out in (BF16, F32):
        assert _run(c, out, 1.0, 1.0, True, act) == g.PATH_SKINNY


@pytest.mark.parametrize("act", [g.ACT_RELU, g.ACT_GELU])
def test_bf16_generic(cuda_lib, act):
    c = inputs.make("decode_m16_o", M=100, N=120, K=88)
    assert _run(c, BF16, 1.0, 1.0, True, act, path=g.PATH_GENERIC) == g.PATH_GENERIC


def test_bad_epilogue_arguments(cuda_lib):
    x = torch.zeros(4096, device="cuda")
    p = x.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32_ex(4, 4, 4, 1.0, p, 4, p, 4, 0.0, p, 4, None, 9, s)
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32_ex(4, 4, 4, 1.0, p, 4, p, 4, 0.0, p, 4, p + 2, 1, s)
    assert e.value.code == g.GEMM_ERR_MISALIGNED
