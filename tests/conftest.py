import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library binding; GPU tests fail loudly if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a CUDA device")
    import transformer_scaled_dot_sdpa_gb300 as g
    return g


# attention kernel schedules (attn_schedule_t): every parity test that uses
# this fixture runs once per schedule
SCHEDULES = {"two_qtiles": 1, "split_keys": 2}


@pytest.fixture(params=list(SCHEDULES.values()), ids=list(SCHEDULES))
def schedule(request, cuda_lib):
    cuda_lib.set_schedule(request.param)
    yield request.param
    cuda_lib.set_schedule(cuda_lib.SCHEDULE_AUTO)
