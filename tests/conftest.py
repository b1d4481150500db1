import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of host time)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


_PARITY_LOG = []


@pytest.fixture(scope="session")
def parity_log():
    """Tests append (name, summary) of full-size comparisons; printed at the end of
    the session (compared / flagged / mismatched positions per workload)."""
    return _PARITY_LOG


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if not _PARITY_LOG:
        return
    tr = terminalreporter
    tr.section("parity at scale (compared / flagged / mismatched)")
    for name, s in _PARITY_LOG:
        parts = []
        for key in ("topk", "walk"):
            if key in s:
                r = s[key]
                parts.append(f"{key} {r['compared']}/{r['flagged']}/{r['mismatched']}")
                if "max_val_rel_err" in r:
                    parts.append(f"max value error {r['max_val_rel_err']:.2e} of max(|v|, 1)")
        for key in ("teacher_forced_rows", "conv_rows", "uniform_rows", "near_tie_rows"):
            if key in s:
                parts.append(f"{key} {s[key]}")
        tr.write_line(f"{name}: " + ", ".join(parts) + ("" if s.get("ok", True) else "  FAILED"))
