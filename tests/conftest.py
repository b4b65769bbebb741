import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_addoption(parser):
    parser.addoption("--kernel-options", default="",
                     help="engram_kernel_options for the whole run, e.g. projection_cta=1,fp8_pair=1")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running test")


@pytest.fixture(autouse=True, scope="session")
def _kernel_options(request):
    """Applies --kernel-options (alternative kernels) before the first test."""
    spec = request.config.getoption("--kernel-options")
    if spec:
        import hashed_gram_conditional_gb300 as eg
        eg.set_kernel_options(**{k: int(v) for k, v in (kv.split("=") for kv in spec.split(","))})
    yield
