"""CUDA-graph capture of library calls.  The entry points neither synchronise
nor allocate, so a sequence of calls captured once on a stream replays as a
graph.  Replays must give the same bits as the same calls launched one by one,
including the launches that overlap through programmatic dependent launch
(the decode kernel, the FP32 kernel's split last wave), also after new operand
values are copied into the captured buffers.  Each kernel family runs once
before the capture: the first call on a device sets kernel attributes and
queries occupancy."""
import pytest
import torch

import roofline_driven_optimisation_gb300 as g
from roofline_driven_optimisation_gb300 import inputs

pytestmark = pytest.mark.gpu
F32, BF16 = torch.float32, torch.bfloat16


def _dev(t):
    return t.cuda()


@pytest.fixture()
def ops(cuda_lib):
    f = inputs.make("fp32_4096", M=2560, N=2048, K=1024)      # 320 tiles: split last wave
    e = inputs.make("fp32_4096", M=300, N=264, K=1024)        # split, bias + GELU
    x = inputs.make("decode_m16_o", M=256, N=4096, K=4096)   # CTA-pair bf16 GEMM
    d = inputs.make("decode_m16_o")                           # 16 x 4096 x 4096, beta 1
    sw = inputs.make_swiglu(16, 1024, 4096)
    t = dict(A1=_dev(f.A), B1=_dev(f.B), C1_0=_dev(f.C0), C1=torch.empty_like(_dev(f.C0)),
             A4=_dev(e.A), B4=_dev(e.B), C4=torch.empty(300, 264, device="cuda"),
             bias=_dev(inputs.random_matrix(1, 264, 77, dist="normal").reshape(264)),
             X=_dev(x.A), W=_dev(x.B), Y=torch.empty(256, 4096, dtype=BF16, device="cuda"),
             W2=_dev(d.B), C3_0=_dev(d.C0), C3=torch.empty_like(_dev(d.C0)),
             Wg=_dev(sw.Bgate), Wu=_dev(sw.Bup),
             S=torch.empty(16, 1024, dtype=BF16, device="cuda"))
    return t


def _sequence(t):
    t["C1"].copy_(t["C1_0"])
    g.gemm(t["A1"], t["B1"], t["C1"], 1.5, 0.5)
    g.gemm(t["A4"], t["B4"], t["C4"], 1.0, 0.0, bias=t["bias"], act=g.ACT_GELU)
    g.gemm(t["X"], t["W"], t["Y"], 1.0, 0.0)
    # the decode GEMM reads rows the previous call wrote
    t["C3"].copy_(t["C3_0"])
    g.gemm(t["Y"][:16], t["W2"], t["C3"], 1.0, 1.0)
    g.swiglu(t["Y"][:16], t["Wg"], t["Wu"], t["S"])


OUTS = ("C1", "C4", "Y", "C3", "S")


def _eager(t):
    _sequence(t)
    torch.cuda.synchronize()
    return {k: t[k].clone() for k in OUTS}


def _replay(gr, t):
    for k in OUTS:
        t[k].fill_(float("nan"))
    gr.replay()
    torch.cuda.synchronize()
    return {k: t[k].clone() for k in OUTS}


def test_graph_replay_matches_eager_calls(ops):
    t = ops
    want = _eager(t)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        _sequence(t)
    torch.cuda.synchronize()
    for _ in range(2):
        got = _replay(gr, t)
        for k in OUTS:
            assert torch.isfinite(got[k]).all(), k
            assert torch.equal(got[k], want[k]), k
    # new values in the captured operand buffers
    t["A1"].copy_(torch.flip(t["A1"], dims=(0,)))
    t["X"].copy_(torch.flip(t["X"], dims=(1,)))
    want2 = _eager(t)
    assert not torch.equal(want2["Y"], want["Y"])
    got = _replay(gr, t)
    for k in OUTS:
        assert torch.equal(got[k], want2[k]), k
    assert g.device_status()[0] == 0
