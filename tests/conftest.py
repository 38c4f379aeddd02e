"""Shared pytest configuration: the ``gpu`` marker and import paths."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity cases (GPU)")


# Every output the binding allocates starts as NaN (E4M3 codes as 0xFF), so an
# element a kernel leaves unwritten fails the parity checks instead of passing
# on whatever the memory held.
from exact_io_aware_21_gb300 import binding as _binding  # noqa: E402

_binding.OUTPUT_CANARY = float("nan")
