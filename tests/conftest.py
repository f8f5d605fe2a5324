import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def _cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Slack statistics of the parity checks that ran (see tests/harness.py): per check,
    the number of calls, elements, the largest flagged fraction, the largest max(slack)/rms
    and the elements whose GPU value differed from the oracle's (all inside the slack)."""
    try:
        from harness import SLACK_RECORDS
    except ImportError:
        return
    if not SLACK_RECORDS:
        return
    agg = {}
    for r in SLACK_RECORDS:
        a = agg.setdefault(r["name"], dict(calls=0, n=0, flagged=0.0, srms=0.0, moved=0))
        a["calls"] += 1
        a["n"] += r["n"]
        a["flagged"] = max(a["flagged"], r["flagged"])
        a["srms"] = max(a["srms"], r["max_slack_rms"])
        a["moved"] += r["moved"]
    tr = terminalreporter
    tr.write_sep("-", "parity slack (per check: calls, elements, max flagged fraction, "
                      "max slack/rms, elements that differ within slack)")
    for name in sorted(agg):
        a = agg[name]
        tr.write_line("%-34s %4d %12d %8.4f %9.5f %10d" % (name, a["calls"], a["n"],
                                                          a["flagged"], a["srms"], a["moved"]))
