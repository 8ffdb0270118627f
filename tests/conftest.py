import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on CPU")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle


@pytest.fixture(autouse=True)
def _status_clean_in_checking_build(request):
    """With NM_LIBRARY naming another build (the bounds-checking one), every GPU
    test must leave the device status word clean: no index out of its buffer,
    no bounded wait run out."""
    yield
    if os.environ.get("NM_LIBRARY") and request.node.get_closest_marker("gpu"):
        import sparse_decoding_gb300 as nm
        st = nm.device_status()
        assert st == nm.NM_OK, f"device status after the test: {nm.status_str(st)}"
