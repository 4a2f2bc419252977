import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The tests load the test build of the engine (libadp_test.so), which also exports the test-only
# hooks; the benchmark and applications load the release build (libadp.so).
os.environ["ADP_TEST_HOOKS"] = "1"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the engine's kernels")
    config.addinivalue_line("markers", "slow: full-size workload; minutes of CPU time")
