import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(autouse=True)
def _no_access_outside_its_buffer(request):
    """With DSV4KV_CHECKED=1 the whole suite runs on the bounds-checked library: after
    every GPU test, no access may have been skipped for leaving its buffer."""
    yield
    if os.environ.get("DSV4KV_CHECKED") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import kv_norm_rope_gb300 as k
    flags = k.debug_bounds_flags(reset=True)
    assert flags == 0, f"checked build: an access outside its buffer was skipped (flags {flags})"
