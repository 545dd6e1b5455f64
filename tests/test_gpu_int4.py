"""INT4 dequantisation through the C ABI, bit for bit against the oracle:
W = scales[k // G][n] * (q - z), exact in fp32 and rounded once to bf16, so
both sides produce identical bits."""
import numpy as np
import pytest
import torch

import roofline_driven_optimisation_gb300 as g
from oracle import int4
from roofline_driven_optimisation_gb300 import inputs

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32


def _expected(c, out, rows=None):
    if rows is None:
        q, sc = c.q, c.scales
        ref = int4.dequant_bf16(q, sc, c.N, c.group, c.zero) if out == BF16 else \
            torch.from_numpy(int4.dequant_exact(q, sc, c.N, c.group, c.zero)).float()
        return ref
    # selected rows k: their groups' scales
    q = c.q[rows]
    sc = c.scales[torch.as_tensor(rows) // c.group]
    ref = int4.dequant_bf16(q, sc, c.N, 1, c.zero) if out == BF16 else \
        torch.from_numpy(int4.dequant_exact(q, sc, c.N, 1, c.zero)).float()
    return ref


def _run(c, out, *, ldq_pad=0, ldw_pad=0, q_off=0):
    K = c.q.shape[0]
    bpr = c.q.shape[1]
    ldq = bpr + ldq_pad
    flat = torch.zeros(q_off + K * ldq + 16, dtype=torch.uint8)
    flat[q_off:q_off + K * ldq].view(K, ldq)[:, :bpr] = c.q
    qd = flat.cuda()
    sd = c.scales.cuda()
    ldw = c.N + ldw_pad
    Wd = torch.full((K, ldw), float("nan"), dtype=out, device="cuda")
    fn = g.gemm_int4_dequant if out == BF16 else g.gemm_int4_dequant_f32
    fn(qd.data_ptr() + q_off, K, c.N, ldq, sd.data_ptr(), c.scales.shape[1], c.group, c.zero,
       Wd.data_ptr(), ldw, torch.cuda.current_stream().cuda_stream)
    ran = g.last_path()
    torch.cuda.synchronize()
    W = Wd.cpu()
    if ldw_pad:
        assert torch.isnan(W[:, c.N:].float()).all()
    return W[:, :c.N].contiguous(), ran


def _same_bits(a, b):
    if a.dtype == BF16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("out", [BF16, F32])
# groups 128, 32 and 4096 run 16 rows per thread, 24 runs 8, 100 runs 4, and 1 the
# 32-codes-per-thread kernel
@pytest.mark.parametrize("group,zero", [(128, 8), (1, 0), (32, 15), (24, 5), (100, 8), (4096, 3)])
def test_vector_kernel_bit_exact(cuda_lib, out, group, zero):
    c = inputs.make_int4(384, 512, group=group, zero=zero, seed=group + zero)
    W, ran = _run(c, out)
    assert ran == g.PATH_INT4
    assert _same_bits(W, _expected(c, out))


@pytest.mark.parametrize("out", [BF16, F32])
@pytest.mark.parametrize("N,ldq_pad,ldw_pad,q_off", [(90, 0, 0, 0), (64, 3, 0, 0), (64, 0, 0, 1),
                                                     (96, 0, 3, 0), (30, 0, 0, 0)])
def test_byte_kernel_bit_exact(cuda_lib, out, N, ldq_pad, ldw_pad, q_off):
    # N not a multiple of 32, rows of q or W not 16-byte aligned: the per-byte kernel
    c = inputs.make_int4(77, N, group=16, zero=8, seed=N)
    W, ran = _run(c, out, ldq_pad=ldq_pad, ldw_pad=ldw_pad, q_off=q_off)
    assert ran == g.PATH_GENERIC
    assert _same_bits(W, _expected(c, out))


def test_odd_column_count(cuda_lib):
    # odd N: the high nibble of each row's last byte is padding and is not written
    c = inputs.make_int4(40, 64, group=8, zero=8, seed=5)
    c.N = 63
    c.scales = c.scales[:, :63].contiguous()
    W, ran = _run(c, BF16, ldw_pad=1)
    assert ran == g.PATH_GENERIC
    assert _same_bits(W, _expected(c, BF16))


@pytest.mark.parametrize("K,out", [(130, BF16), (144, BF16), (144, F32)])
def test_padded_vector_rows(cuda_lib, K, out):
    # K = 130 takes the 32-codes-per-thread kernel, K = 144 the row-blocked one
    c = inputs.make_int4(K, 256, group=48, zero=8, seed=3)
    W, ran = _run(c, out, ldq_pad=16, ldw_pad=8)
    assert ran == g.PATH_INT4
    assert _same_bits(W, _expected(c, out))


def test_long_by_long_sampled(cuda_lib):
    # the 16384 x 16384 matrix of the benchmark, checked on sampled rows
    c = inputs.make_int4(16384, 16384, group=128, zero=8, seed=8)
    W = torch.empty((16384, 16384), dtype=BF16, device="cuda")
    g.int4_dequant(c.q.cuda(), c.scales.cuda(), 16384, 128, 8, W)
    torch.cuda.synchronize()
    assert g.last_path() == g.PATH_INT4
    rows = sorted({0, 1, 127, 128, 8191, 16383, *np.random.default_rng(1).choice(16384, 10).tolist()})
    assert _same_bits(W[rows].cpu(), _expected(c, BF16, rows))


def test_arguments(cuda_lib):
    q = torch.zeros((4, 8), dtype=torch.uint8, device="cuda")
    s = torch.ones((1, 16), dtype=BF16, device="cuda")
    W = torch.zeros((4, 16), dtype=BF16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for args, code in (((4, 16, 8, 16, 0, 8), g.GEMM_ERR_INVALID_ARG),     # group 0
                       ((4, 16, 8, 16, 4, 16), g.GEMM_ERR_INVALID_ARG),    # zero 16
                       ((4, 16, 7, 16, 4, 8), g.GEMM_ERR_INVALID_ARG)):    # ldq < N/2
        K, N, ldq, lds, group, zero = args
        with pytest.raises(g.GemmError) as e:
            g.gemm_int4_dequant(q.data_ptr(), K, N, ldq, s.data_ptr(), lds, group, zero,
                                W.data_ptr(), 16, st)
        assert e.value.code == code
    with pytest.raises(g.GemmError) as e:
        g.gemm_int4_dequant(q.data_ptr(), 4, 16, 8, s.data_ptr() + 1, 16, 4, 8, W.data_ptr(), 16, st)
    assert e.value.code == g.GEMM_ERR_MISALIGNED
    g.gemm_int4_dequant(None, 0, 16, 8, None, 16, 4, 8, None, 16, st)   # K = 0: no-op
    # all codes equal to the zero point give exact zeros
    q.fill_(0x88)
    g.gemm_int4_dequant(q.data_ptr(), 4, 16, 8, s.data_ptr(), 16, 4, 8, W.data_ptr(), 16, st)
    torch.cuda.synchronize()
    assert torch.equal(W.float().cpu(), torch.zeros((4, 16)))
