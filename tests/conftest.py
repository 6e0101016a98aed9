import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity cases")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print what the GPU parity tests measured (intermediate code match, FP8
    scale deviations), pass or fail."""
    try:
        from gpu_util import REPORT
    except Exception:
        return
    if REPORT:
        terminalreporter.section("parity measurements")
        for line in REPORT:
            terminalreporter.write_line(line)
