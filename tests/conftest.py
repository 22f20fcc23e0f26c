import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")
    config.addinivalue_line("markers", "ue8m0: a GPU case with UE8M0 scales that runs on both m-grouped kernels")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _debug_word_stays_clear(request):
    """With DG_DEBUG=1 (the debug build, whose kernels check every index they compute), every GPU
    test must leave the debug word clear: no kernel computed an index outside its buffers."""
    yield
    if os.environ.get("DG_DEBUG") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    from moe_grouped_fp8_gb300 import api
    word = api.dg_debug_word(clear=True)
    assert word == 0, f"debug build: index check bits {word:#x} raised during {request.node.nodeid}"
