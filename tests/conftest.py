import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# the library's test hooks (tile widths, schedules, fault injection) answer
# only in a process that enables them
os.environ["FP8RL_TEST_HOOKS"] = "1"
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")
