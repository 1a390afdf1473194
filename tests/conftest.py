import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running parity case")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Raw parity figures of every GPU-vs-oracle comparison made in this run
    (max |err|, relative Frobenius error and max |ref| per tensor)."""
    parity = sys.modules.get("parity")
    if parity is None or not getattr(parity, "REPORT", None):
        return
    terminalreporter.section("parity against the float64 oracle (raw errors)")
    for line in parity.format_report():
        terminalreporter.write_line(line)
