import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (full-size) case")


@pytest.fixture(autouse=True)
def _no_out_of_bounds_access(request):
    """With the bounds-checked build loaded (ZERO_LIB=.../libzero_checked.so),
    every GPU test must end without a kernel access outside the extents its
    layout gives: the checked kernels skip and count such accesses."""
    yield
    if not os.environ.get("ZERO_LIB") or request.node.get_closest_marker("gpu") is None:
        return
    from zero_partitioned_mixed_replica_gb300 import binding as B
    if B.zero_checked_build():
        assert B.zero_bounds_violations(reset=True) == 0, "a kernel skipped an out-of-bounds access"
