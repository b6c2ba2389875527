import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """After every GPU test: no kernel of the library gave up a bounded wait (QMM_ERR_TIMEOUT) and, with
    the library built with QMM_DEBUG (QMM_DEBUG=1 in the environment), no device bounds check failed
    (QMM_ERR_BOUNDS)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch

    if not torch.cuda.is_available():
        return
    import block_quantized_matmul_gb300 as qmm

    torch.cuda.synchronize()
    st = qmm.qmm_device_status()
    assert st == 0, f"device status {qmm._STATUS.get(st, st)} after this test"
