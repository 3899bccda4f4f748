import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    from flag_report import RESULTS
    if not RESULTS:
        return
    terminalreporter.write_line("parity: sequences compared in full / flagged (near-tie decisions)")
    for case, (compared, flagged) in sorted(RESULTS.items()):
        detail = "; ".join(f"seq {b}: {why}" for b, why in flagged)
        terminalreporter.write_line(f"  {case}: {compared} compared, {len(flagged)} flagged"
                                    + (f" ({detail})" if detail else ""))
