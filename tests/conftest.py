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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of host work")


@pytest.fixture(autouse=True)
def _device_index_checks(request):
    """Under the MHC_CHECK build (MHC_GB300_CHECK=1), every GPU test also
    asserts that no device index check failed while it ran."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    if os.environ.get("MHC_GB300_CHECK", "0") in ("", "0"):
        return
    import gemm_rms_sinkhorn_gb300 as mhc

    site, off, extent = mhc.mhc_testing_check_record()
    assert site == 0, "device index check %d failed: offset %d of %d" % (site, off, extent)
