import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


# Every GPU test runs with the batch-invariant limit covering any size it uses, so that the
# invariant kernels are the ones under test; a test of the non-invariant path sets the
# limit itself inside this fixture's scope, and the previous value is restored after it.
INVARIANT_EVERYWHERE = 1 << 40


@pytest.fixture(autouse=True)
def _batch_invariant_limit(request):
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    try:
        import invariant_bi_matmul_gb300 as bi
        old = bi.get_batch_invariant_limit()
    except Exception:  # library not built: the test itself reports that
        yield
        return
    bi.set_batch_invariant_limit(INVARIANT_EVERYWHERE)
    try:
        yield
    finally:
        bi.set_batch_invariant_limit(old)
