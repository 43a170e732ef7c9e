import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


import pytest


@pytest.fixture(autouse=True)
def _no_device_timeout(request):
    """After every GPU test: no bounded device-side wait of the library ran out."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from weight_only_quantized_qgemv_gb300 import _lib
    status = _lib.qdevice_error(clear=True)
    assert status == 0, f"device wait timed out during the test: {_lib.qstatus_string(status)}"
