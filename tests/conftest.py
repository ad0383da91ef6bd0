import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(autouse=True)
def _no_failed_bounds_checks(request):
    """With QGEMV_BOUNDS_CHECK=1 the binding loads the bounds-checking build:
    then every GPU test must also leave no failed index check behind (the
    records are read, and cleared, after the test)."""
    yield
    if os.environ.get("QGEMV_BOUNDS_CHECK", "0") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    if "test_gpu_bounds_check" in request.node.nodeid:  # plants a failure on purpose, in a child process
        return
    import torch

    if not torch.cuda.is_available():
        return
    from block_quantized_gemv_quantize_gb300 import ops

    count, site = ops.qgemv_take_bounds_errors()
    assert count == 0, f"{count} failed bounds checks, the first at site {site}"
