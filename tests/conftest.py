import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def orc():
    """The CPU oracle package, built on first use."""
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(params=["fast", "exact"])
def statistic(request):
    """Runs the test under each row statistic of the modulating operations
    (restoring the previous one after it)."""
    import diffusion_transformer_elementwise_gb300 as dit
    with dit.statistic(request.param):
        yield request.param
