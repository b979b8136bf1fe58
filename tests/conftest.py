import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_sessionstart(session):
    # build (or confirm up to date) the CUDA library and the C oracle; both
    # builds are no-ops when nothing changed
    from qk_rmsnorm_rope_gb300 import build as qknr_build
    qknr_build.build()
    import oracle
    oracle.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()
