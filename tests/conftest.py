import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); run with -m gpu")
    # compile whatever native part is missing or older than its sources (the CUDA
    # library, the device input generator, the C oracle); nothing when up to date
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="session")
def ora():
    import oracle
    return oracle.load()


@pytest.fixture(autouse=True)
def _device_status_stays_clear(request):
    """Every GPU test ends with the device status word clear: no bounded wait of
    the TMA form ran out (a block that gives up leaves its chunks unprocessed)."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    try:
        import torch
        if not torch.cuda.is_available():
            yield
            return
        import fully_sharded_gb300 as fs
    except ImportError:
        yield
        return
    fs.fsdp_device_status(clear=True)
    yield
    assert fs.fsdp_device_status() == 0, "a bounded device wait ran out during this test"
