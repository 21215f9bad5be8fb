import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.lib()
    return o


@pytest.fixture(scope="session")
def bsq():
    """The CUDA library through its Python binding.  On a GPU run a missing or
    unloadable library is a failure, never a skip."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    from block_scaled_precision_packed_gb300 import bsq as b
    b.load()
    return b


@pytest.fixture(autouse=True)
def _clean_device_error_word(request):
    """After every GPU test: no bounded wait timed out and no device check fired."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from block_scaled_precision_packed_gb300 import bsq as b
    st, code = b.device_error()
    assert st == 0 and code == 0, f"device error word set: status {st}, site 0x{code:x}"
