"""The FP32 FMA probe: the roofline's FP32 peak (SMs x 128 lanes x 2 FLOP x
maximum SM clock) bounds what the lanes retire, with scalar and with packed
f32x2 FMAs; a packed rate above the bound would mean the peak definition
undercounts the hardware."""
import pytest
import torch

import bench_probe
from roofline_driven_optimisation_gb300 import roofline as R

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def probe_lib():
    bench_probe.build()
    bench_probe.load()
SM_MAX_HZ = 2070e6


@pytest.mark.parametrize("packed", [False, True])
def test_fma_rate_within_the_fp32_peak(cuda_lib, packed):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    peak = R.fp32_peak(sms, SM_MAX_HZ)
    sink = torch.zeros(1, device="cuda")
    s = torch.cuda.current_stream()
    bench_probe.probe_fp32_fma(packed, 2000, sink.data_ptr(), s.cuda_stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    flops = bench_probe.probe_fp32_fma(packed, 8000, sink.data_ptr(), s.cuda_stream)
    e1.record(s)
    torch.cuda.synchronize()
    assert flops == sms * 4 * 256 * 8000 * 16 * 2 * 2
    rate = flops / (e0.elapsed_time(e1) * 1e-3)
    assert rate <= 1.02 * peak, f"{rate / 1e12:.1f} TFLOP/s above the {peak / 1e12:.1f} peak"
    assert rate >= 0.5 * peak
    assert sink.item() == 0.0


def test_probe_rejects_bad_arguments(cuda_lib):
    with pytest.raises(ValueError):
        bench_probe.probe_fp32_fma(True, 0, 0)
