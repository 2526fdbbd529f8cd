import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU check")


def pytest_terminal_summary(terminalreporter):
    """After a GPU run: the worst per-tensor and per-row errors of each compared quantity
    against its tolerance, and the discrete decisions of each workload variant against the
    fp64 oracle's own (rounds, flagged near-ties, unflagged disagreements)."""
    h = sys.modules.get("gpu_harness")
    if h is None or not (h.MARGINS or h.DECISIONS):
        return
    tr = terminalreporter
    tr.write_sep("-", "parity margins: worst rel err per tensor / per row (tolerance)")
    for name, (e, r, tol) in sorted(h.MARGINS.items()):
        tr.write_line(f"{name}: {e:.2e} / {r:.2e} ({tol:g})")
    tr.write_sep("-", "decisions vs the fp64 oracle (per sequence-round)")
    for name, rec in sorted(h.DECISIONS.items()):
        tr.write_line(f"{name}: rounds={rec['rounds']} near_ties={rec['near_ties']} "
                      f"fp64_disagreements={rec['fp64_disagreements']} "
                      f"(on flagged near-ties: {rec['near_tie_disagreements']})")
