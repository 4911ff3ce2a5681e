import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdflash.so")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(autouse=True)
def device_status_stays_clear(request):
    """Every GPU test starts with the library's device status clear and must
    leave it clear: a bounded wait that gave up (DFLASH_DEV_TIMEOUT) or an
    input flagged by a kernel fails the test that caused it.  Tests that
    provoke a status bit read it (which clears it) themselves."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import block_speculative_decoding_gb300 as dfl
    dfl.read_device_status()
    yield
    st = dfl.read_device_status()
    assert st == 0, "device status 0x%x left set by this test" % st
