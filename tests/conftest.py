import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _build_library():
    """Build libq8ta.so in-tree when a source is newer (a no-op otherwise)."""
    import shutil
    if shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc"):
        from int8_quantized_q8ta_gb300 import _build
        _build.build()


def pytest_configure(config):
    _build_library()
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU case")
