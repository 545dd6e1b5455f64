"""Attention through the C ABI against the fp64 oracle.  Error scale: the
largest sum_j P[i][j] |V[j][c]| (each output element is that weighted average
of V, rounded).  Tolerance 6e-3: P is rounded to bf16 before the second
product and O once more at the end, each at most 2^-9 of that scale, plus the
fp32 accumulation and the exp2 approximation."""
import numpy as np
import pytest
import torch

import oracle
import roofline_driven_optimisation_gb300 as g
from oracle import attention as A
from roofline_driven_optimisation_gb300 import inputs

pytestmark = pytest.mark.gpu
TOL = 6e-3


def _run(c, causal=False, scale=0.0, path=None):
    Q, K, V = c.Q.cuda(), c.K.cuda(), c.V.cuda()
    O = torch.full_like(Q, float("nan"))
    if path is not None:
        g.force_path(path)
    try:
        g.attention(Q, K, V, O, scale=scale, causal=causal)
        ran = g.last_path()
    finally:
        g.force_path(g.PATH_AUTO)
    torch.cuda.synchronize()
    status, where = g.device_status()
    assert status == 0, f"device status {status} at site {where}"
    return O.cpu(), ran


def _check(c, causal=False, scale=0.0, **kw):
    O, ran = _run(c, causal, scale, **kw)
    sc = scale if scale else None
    ref = A.attention(c.Q, c.K, c.V, sc, causal)
    den = A.error_scale(c.Q, c.K, c.V, sc, causal)
    err = oracle.normwise_error(O, ref, den if den else 1.0)
    assert err <= TOL, f"normwise error {err:.3e} > {TOL} (path {g.PATH_NAMES.get(ran)})"
    return err, ran


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [128, 256, 200, 64, 1])
def test_self_attention(cuda_lib, D, causal, S):
    c = inputs.make_attention(B=2, Hq=3, Hkv=3, Sq=S, Sk=S, D=D, seed=S + D)
    _, ran = _check(c, causal)
    assert ran == g.PATH_ATTN


@pytest.mark.parametrize("Sq,Sk,causal", [(64, 300, True), (300, 64, True), (130, 517, False),
                                          (1, 1000, True), (257, 129, False)])
def test_unequal_lengths(cuda_lib, Sq, Sk, causal):
    # the causal alignment puts the last query at the last key: with Sq > Sk
    # the first Sq - Sk rows see no key and are 0
    c = inputs.make_attention(B=1, Hq=2, Hkv=2, Sq=Sq, Sk=Sk, D=128, seed=Sq + Sk)
    _, ran = _check(c, causal)
    assert ran == g.PATH_ATTN


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("Sq,Sk,causal", [(700, 700, True), (700, 700, False), (1000, 700, True),
                                          (384, 1200, True), (640, 333, False)])
def test_several_query_blocks_and_key_tiles(cuda_lib, D, Sq, Sk, causal):
    # query blocks of two 128-row tiles, ragged last block (its second tile
    # may lie past Sq), several 128-key tiles with a ragged last one
    c = inputs.make_attention(B=1, Hq=2, Hkv=1, Sq=Sq, Sk=Sk, D=D, seed=Sq + 3 * Sk + D)
    _, ran = _check(c, causal)
    assert ran == g.PATH_ATTN


@pytest.mark.parametrize("D", [128, 64])
def test_causal_tiles_outnumber_resident_ctas(cuda_lib, D):
    # 8 query tiles x 80 heads = 640 CTAs, more than fit on the GPU at once:
    # the longest-first causal dispatch runs in waves of tiles of different
    # lengths, with grouped key/value heads; every output row checked
    c = inputs.make_attention(B=2, Hq=40, Hkv=8, Sq=1000, Sk=1000, D=D, seed=41 + D)
    _, ran = _check(c, True)
    assert ran == g.PATH_ATTN


def test_causal_tiles_without_keys_among_many_ctas(cuda_lib):
    # Sq > Sk: the first three query tiles of every head see no key, so their
    # CTAs load nothing and issue no MMA but still write zero rows, among
    # 640 CTAs that do (10 query tiles x 64 heads)
    c = inputs.make_attention(B=1, Hq=64, Hkv=8, Sq=1200, Sk=700, D=128, seed=43)
    _, ran = _check(c, True)
    assert ran == g.PATH_ATTN


def test_grouped_kv_heads_and_scale(cuda_lib):
    c = inputs.make_attention(B=2, Hq=8, Hkv=2, Sq=192, Sk=320, D=128, seed=3)
    _check(c, True)
    _check(c, False, scale=0.05)


def test_large_scores_stay_finite(cuda_lib):
    # scores around +-200 (scale 1): the online maximum must keep exp2 finite
    c = inputs.make_attention(B=1, Hq=2, Hkv=2, Sq=256, Sk=384, D=128, seed=4)
    c.Q = (c.Q.float() * 2).to(torch.bfloat16)
    _check(c, True, scale=1.0)


@pytest.mark.parametrize("D", [32, 96])
def test_generic_head_dims(cuda_lib, D):
    c = inputs.make_attention(B=1, Hq=2, Hkv=1, Sq=70, Sk=90, D=D, seed=D)
    for causal in (False, True):
        _, ran = _check(c, causal)
        assert ran == g.PATH_GENERIC


def test_forced_generic_agrees(cuda_lib):
    c = inputs.make_attention(B=1, Hq=2, Hkv=2, Sq=256, Sk=256, D=128, seed=6)
    _, ran = _check(c, True, path=g.PATH_GENERIC)
    assert ran == g.PATH_GENERIC


def test_deterministic(cuda_lib):
    c = inputs.make_attention(B=1, Hq=4, Hkv=4, Sq=384, Sk=384, D=128, seed=7)
    a, _ = _run(c, True)
    b, _ = _run(c, True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_llama_prefill_layer_sampled(cuda_lib):
    # one LLaMA-7B layer's prefill (32 heads of 128, 2048 tokens, causal),
    # checked on three heads against the oracle
    c = inputs.make_attention()
    O, ran = _run(c, True)
    assert ran == g.PATH_ATTN
    for h in (0, 17, 31):
        sub = inputs.AttentionCase(c.Q[:, h:h + 1], c.K[:, h:h + 1], c.V[:, h:h + 1])
        ref = A.attention(sub.Q, sub.K, sub.V, None, True)
        den = A.error_scale(sub.Q, sub.K, sub.V, None, True)
        err = oracle.normwise_error(O[:, h:h + 1], ref, den)
        assert err <= TOL, (h, err)


def test_arguments(cuda_lib):
    q = torch.zeros((1, 3, 8, 64), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 2, 8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemmError) as e:      # 3 query heads over 2 kv heads
        g.gemm_attention(1, 3, 2, 8, 8, 64, q.data_ptr(), kv.data_ptr(), kv.data_ptr(), q.data_ptr(), 0.0, 0,
                         torch.cuda.current_stream().cuda_stream)
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_attention(1, 2, 2, 8, 8, 64, q.data_ptr(), kv.data_ptr(), kv.data_ptr(), q.data_ptr(), -1.0, 0,
                         torch.cuda.current_stream().cuda_stream)
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    g.gemm_attention(0, 2, 2, 8, 8, 64, None, None, None, None, 0.0, 0, 0)   # B = 0: nothing to do
