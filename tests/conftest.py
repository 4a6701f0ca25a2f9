import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when the GPU or the library is missing;
    # nothing to adjust here beyond the markers.
    return
