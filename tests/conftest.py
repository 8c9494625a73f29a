import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103) and the built CUDA library")


def fp32_tolerance(ref):
    """Acceptance bound for uniform inputs: |C_gpu - C_ref| <= 1e-3 + 1e-3*|C_ref|."""
    import numpy as np
    return 1e-3 + 1e-3 * np.abs(ref)
