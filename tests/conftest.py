import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library (only for tests marked gpu)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import roofline_driven_optimisation_gb300 as g
    g.load()
    return g
