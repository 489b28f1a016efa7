import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large inputs")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture
def testing_build():
    """Route the library calls of one test to the testing build (the one with
    the debug hooks), with every hook at its default before and after."""
    import bwd_gn3d_stats_gb300 as gn
    from bwd_gn3d_stats_gb300 import build

    build.build()
    defaults = {gn.DEBUG_PATH: 0, gn.DEBUG_LAG: -1, gn.DEBUG_SLOTS: -1, gn.DEBUG_SPIN_LIMIT: 0,
                gn.DEBUG_SHARES: -1, gn.DEBUG_RES_HELD: -1, gn.DEBUG_RES_WINDOW: -1, gn.DEBUG_RES_PASS: -1,
                gn.DEBUG_FAIL_NEXT: 0, gn.DEBUG_FORCE_TIMEOUT: 0}
    prev = gn.use_library("testing")
    for k, v in defaults.items():
        gn.gn3d_debug_set(k, v)
    try:
        yield gn
    finally:
        for k, v in defaults.items():
            gn.gn3d_debug_set(k, v)
        gn.use_library(prev)
