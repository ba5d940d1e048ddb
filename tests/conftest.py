import contextlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture
def tune():
    """tune(**fields) installs library layout overrides (sscan_set_tuning) for the rest of the
    test; each call replaces the previous setting; teardown restores the automatic choices."""
    from selective_state_space_158_b300 import binding

    stack = contextlib.ExitStack()

    def set_(**fields):
        stack.enter_context(binding.tuning(**fields))

    yield set_
    stack.close()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (parity tests through the C ABI)")
    config.addinivalue_line("markers", "slow: long-running CPU test")
