import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU check")


@pytest.fixture(scope="session", autouse=True)
def _native_build():
    """Build the in-tree native libraries and the CPU checker once per session."""
    from fsdp_sharded_mixed_shard_gb300 import _build
    import oracle.build
    _build.build()
    oracle.build.build()
    yield
