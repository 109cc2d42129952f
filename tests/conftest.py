import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA device (GB300, sm_103a); parity through the C ABI")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, loaded through the Python binding."""
    from differential_attention_diff_gb300 import binding
    return binding.load()
