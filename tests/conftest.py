import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture
def pkv_opts():
    """Setter of the library's options for one test; the options in force
    before the test are put back afterwards."""
    import paged_kv_cache_195_gb300 as pkv
    saved = pkv.get_options()

    def set_(**changes):
        pkv.set_options(**changes)

    yield set_
    pkv.set_options(**saved)
