import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libnvfp4.so")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(autouse=True)
def _bounds_record_clean(request):
    """Under the bounds-checked build (NVFP4_LIB=checked) every GPU test must
    leave no failed address test behind: any kernel access outside the
    shared-memory window, the TMEM columns or the bytes its call's arguments
    grant fails the test that made it."""
    yield
    if os.environ.get("NVFP4_LIB") != "checked" or request.node.get_closest_marker("gpu") is None:
        return
    import nvfp4_block_scaled_30_b300 as nv
    if nv._LIB is None:
        return
    n, where, value, limit = nv.bounds_record(clear=True)
    assert n == 0, f"{n} failed address tests; the first at {where}: value {value}, limit {limit}"
