"""Abort paths of the real kernels (failure detection without a GPU fault).

gemm_test_stall makes one role of the first CTA or cluster wait on a barrier
that nothing arrives at.  Its bounded wait runs out; the kernel records
GEMM_ERR_DEVICE_TIMEOUT with that role's location code, the other roles and
the other CTAs of its cluster leave through the abort path (their copies and
MMAs drained, the cluster barriers reached by every rank, tensor memory
freed), and the context stays usable: the next call, with the hook off, is
checked against the oracle.  Nothing is skipped that could fault: every copy
that was issued lands, and no address changes."""
import pytest
import torch

import roofline_driven_optimisation_gb300 as g
from roofline_driven_optimisation_gb300 import inputs
from gpu_util import check

pytestmark = pytest.mark.gpu

BF16, F32 = torch.bfloat16, torch.float32
# location codes of the stalled roles (the WaitSite values of the library)
SITE_TC2_MMA, SITE_SIMT_CONSUMER, SITE_SKINNY_MMA = 15, 21, 31
LIMIT_NS = 8_000_000     # 8 ms: the stalled wait gives up after 2 ms


@pytest.fixture
def short_limit(cuda_lib):
    assert g.device_status()[0] == 0
    g.set_wait_timeout_ns(LIMIT_NS)
    try:
        yield
    finally:
        g.test_stall(0)
        g.set_wait_timeout_ns(0)
        g.force_tc_pair(0)
        g.force_tile_n(0)


def stalled_call(A, B, C0, alpha, beta, out):
    """One call with the hook on; returns (status, where, family facts)."""
    dev = "cuda"
    M, N = A.shape[0], B.shape[1]
    C = C0.to(out).to(dev) if C0 is not None else torch.zeros((M, N), dtype=out, device=dev)
    g.test_stall(1)
    try:
        g.gemm(A.to(dev), B.to(dev), C, alpha, beta)
    finally:
        g.test_stall(0)
    facts = (g.last_path(), g.last_k_split(), g.last_tc_pair())
    torch.cuda.synchronize()
    status, where = g.device_status()
    return status, where, facts


def test_tc2_pair_abort_then_recovers(short_limit):
    c = inputs.make("bf16_4096", M=512, N=512, K=256)
    g.force_tc_pair(2)
    status, where, (path, _, pair) = stalled_call(c.A, c.B, None, 1.0, 0.0, BF16)
    assert path == g.PATH_BF16_TC and pair in (2, 4, 6)
    assert (status, where) == (g.GEMM_ERR_DEVICE_TIMEOUT, SITE_TC2_MMA)
    assert g.device_status()[0] == 0          # taken once
    err, path = check(c.A, c.B, None, 1.0, 0.0, BF16)
    assert path == g.PATH_BF16_TC and g.last_tc_pair() in (2, 4, 6)


def test_tc2_stream_k_abort_then_recovers(short_limit):
    # every tile in the stream-K tail (6 tiles, 64 K-steps, 48 pairs): the
    # first pair's MMA issuer stalls, so it never hands over its partial
    # tiles; the finishers waiting for them give up and the flags the other
    # pairs raised are lowered when the status is read.  Five later calls
    # (every workspace slot) match the oracle.
    c = inputs.make("bf16_4096", M=300, N=520, K=4096)
    g.force_tc_pair(2)
    g.force_tile_n(256)
    g.force_split_tiles(2)
    try:
        status, where, (path, _, pair) = stalled_call(c.A, c.B, None, 1.0, 0.0, BF16)
        assert path == g.PATH_BF16_TC and pair == 6
        assert (status, where) == (g.GEMM_ERR_DEVICE_TIMEOUT, SITE_TC2_MMA)
        assert g.device_status()[0] == 0
        for _ in range(5):
            check(c.A, c.B, None, 1.0, 0.0, BF16)
            assert g.last_tc_pair() == 6
    finally:
        g.force_split_tiles(1)


def test_skinny_split_abort_then_recovers(short_limit):
    # 2 column slabs, K 4096: the K range is split over a cluster of 8 CTAs
    c = inputs.make("decode_m4_o", M=4, N=256, K=4096)
    status, where, (path, split, _) = stalled_call(c.A, c.B, c.C0, 1.0, 1.0, BF16)
    assert path == g.PATH_SKINNY and split > 1
    assert (status, where) == (g.GEMM_ERR_DEVICE_TIMEOUT, SITE_SKINNY_MMA)
    err, path = check(c.A, c.B, c.C0, 1.0, 1.0, BF16)
    assert path == g.PATH_SKINNY and g.last_k_split() > 1


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("M,N,K", [(300, 260, 1024),     # split launch only (6 or 3 tiles)
                                   (2560, 2048, 1024)])  # whole waves, then the split launch
def test_simt_split_abort_then_recovers(short_limit, bn, M, N, K):
    c = inputs.make("fp32_4096", M=M, N=N, K=K)
    g.force_tile_n(bn)
    try:
        status, where, (path, split, _) = stalled_call(c.A, c.B, c.C0, 1.5, 0.5, F32)
        assert path == g.PATH_F32_SIMT and split > 1 and g.last_tile_n() == bn
        assert (status, where) == (g.GEMM_ERR_DEVICE_TIMEOUT, SITE_SIMT_CONSUMER)
        err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32)
        assert path == g.PATH_F32_SIMT and g.last_k_split() > 1
    finally:
        g.force_tile_n(0)
