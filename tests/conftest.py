import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run with -m gpu on the GPU box)")


def read_golden(name):
    """Parse a `key v1 v2 ...` fixture under tests/golden (comments start with #)."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *vals = line.split()
            nums = [float(v) for v in vals]
            out[k] = nums if len(nums) > 1 else nums[0]
    return out


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The per-case count of near-threshold exclusions from bit-exact parity."""
    try:
        import _report
    except ImportError:
        return
    if not _report.RECORDS:
        return
    tr = terminalreporter
    tr.write_sep("-", "near-threshold exclusions from bit-exact parity (oracle flags within 1e-6)")
    tot_c = tot_f = 0
    for case, compared, flagged, unit in _report.RECORDS:
        tr.write_line("%-60s %6d %-9s compared, %4d flagged (%.2f%%)"
                      % (case[:60], compared, unit, flagged, 100.0 * flagged / max(1, compared)))
        tot_c += compared
        tot_f += flagged
    tr.write_line("%-60s %6d compared, %4d flagged (%.3f%%)" % ("total", tot_c, tot_f, 100.0 * tot_f / max(1, tot_c)))
