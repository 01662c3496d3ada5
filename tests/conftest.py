import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large workload (full K3 sizes)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # the K3-size parity cases' index and error figures (near-ties per config)
    try:
        from parity_util import REPORT
    except Exception:
        return
    if REPORT:
        terminalreporter.section("K3 parity report")
        for line in REPORT:
            terminalreporter.write_line(line)
