import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def fa():
    """The CUDA library's Python binding; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_tcgen05_gb300 as pkg
    pkg.load()          # raises if the compiled library is missing
    return pkg


@pytest.fixture(autouse=True)
def _device_status_after_each_test(request):
    """With FA_GB300_CHECK_STATUS set (the bounds-checking runs), every GPU test
    must leave the device status word clear: a kernel whose index check failed
    records status 7 there instead of touching memory."""
    yield
    if not os.environ.get("FA_GB300_CHECK_STATUS") or "fa" not in request.fixturenames:
        return
    import exact_io_aware_tcgen05_gb300 as pkg
    assert pkg.fa_debug_checks_enabled(), "FA_GB300_CHECK_STATUS set without the checking build"
    pkg.fa_device_status()      # raises on a recorded failed check
