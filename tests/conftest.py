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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (built for sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.lib()
    return oracle


@pytest.fixture(params=[2, 0], ids=["bulk", "plain"])
def bulk(request):
    """Run a GPU test with the insert's bulk-copy pipeline shape for every
    call whose layout qualifies, then with the row-per-warp shape only (both
    must give identical results)."""
    from pack_mla_cache_gb300 import build, ops

    build.build()
    prev = ops.mla_set_bulk_copy(request.param)
    yield request.param
    ops.mla_set_bulk_copy(prev)
