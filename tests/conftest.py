import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU reference computation")
    # every buffer the binding allocates for a test starts as NaN bytes, so an
    # output element the library never writes fails the comparison instead of
    # passing with a value a previous call left in recycled memory
    from folded_tensor_sequence_zigzag_gb300 import tsp
    tsp.POISON = True
