import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_sessionstart(session):
    # Build the CUDA library (nvcc cross-compiles without a GPU) and the
    # oracle before any test imports them.
    path = os.path.join(ROOT, "full_gqa_attention_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_spark_attn_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import oracle
    oracle.build()


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    torch.cuda.set_device(0)
    # calls that allocate their own workspace report device faults too
    import full_gqa_attention_gb300 as fga
    fga.check_device_status(True)
    return torch.device("cuda:0")
