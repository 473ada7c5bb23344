import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def rbkv():
    """The library binding, built in-tree first if stale."""
    from ragged_blocked_kv_gb300 import build as _build
    _build.build()
    import ragged_blocked_kv_gb300 as m
    m.lib()
    return m
