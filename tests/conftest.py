import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")
    config.addinivalue_line("markers", "slow: long-running check")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


# Device waits give up after 0.5 s in tests (default 4 s): a kernel whose
# pipeline bookkeeping is wrong fails its test quickly instead of stalling.
os.environ.setdefault("CONV3D_TIMEOUT_MS", "500")
