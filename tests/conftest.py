import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103) and the built CUDA library")
    config.addinivalue_line(
        "markers", "slow: full-size workload (minutes of CPU oracle work)")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (built on first use)."""
    from packed_sequence_attention_gb300 import _binding
    return _binding.load(build_if_missing=True)
