import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture
def lib_option():
    """Set process-wide library options (ssd_complex_set_option) for one test;
    every option set is put back to its default afterwards."""
    from state_space_sequence_complex_gb300 import ssdc
    touched = set()

    def setter(key, value):
        ssdc.set_option(key, int(value))
        touched.add(key)
    yield setter
    for k in touched:
        ssdc.set_option(k, ssdc.option.DEFAULTS[k])


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built libssdc.so")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")
