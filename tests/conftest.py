import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


@pytest.fixture(scope="session")
def ssm_lib():
    """The CUDA library, built in-tree if missing (nvcc cross-compiles without a GPU)."""
    from selective_state_space_137_b300.build import build_library
    build_library()
    from selective_state_space_137_b300 import binding
    return binding


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("test marked gpu but no CUDA device is visible")
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def device_status_clean(request):
    """After every GPU test, the library's device error word must be clear: a
    kernel whose bounded wait gave up returns normally with its outputs
    incomplete, so a test that passed on such outputs would otherwise hide it.
    (Tests that make a wait run out on purpose read and clear the word.)"""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from selective_state_space_137_b300 import binding
    st = binding.ssm_get_device_status()
    assert st == binding.SSM_OK, f"device error word after the test: {binding.ssm_status_string(st)}"
