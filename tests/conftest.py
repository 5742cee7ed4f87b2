import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Prints the accuracy records of tests.helpers.report: error against the
    float64 oracle, as the worst error/bound ratio and the fraction of
    elements out of bound for the contract tolerance and for the tighter
    Inference Cookbook FAQ Q10 tolerance (reported, not asserted)."""
    try:
        from tests.helpers import ACCURACY
    except Exception:  # pragma: no cover
        return
    if not ACCURACY:
        return
    tr = terminalreporter
    tr.section("accuracy against the float64 oracle (reported, not asserted)")
    tr.line(f"{'result':44s} {'dtype':5s} {'max|err|':>9s} {'contract worst/frac':>22s} "
            f"{'FAQ Q10 worst/frac':>22s}  reference")
    for name, refname, dtype, st in ACCURACY:
        c, p = st["contract"], st["pages_q10"]
        tr.line(f"{name:44s} {dtype:5s} {st['max_abs_err']:9.2e} "
                f"{c['worst_ratio']:10.3f} {c['frac_out']:10.2e} "
                f"{p['worst_ratio']:10.3f} {p['frac_out']:10.2e}  {refname}")
