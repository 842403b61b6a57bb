import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkla.so")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """List every oracle comparison of the run: the scaled error that is
    asserted and the plain relative error beside it."""
    try:
        from helpers import RECORDS
    except ImportError:  # pragma: no cover
        return
    if not RECORDS:
        return
    tr = terminalreporter
    tr.write_sep("-", f"parity against the fp64 oracle ({len(RECORDS)} comparisons)")
    worst = {}
    for what, tol, errs in RECORDS:
        scaled = max((v for k, v in errs.items() if not k.startswith("rel_")), default=0.0)
        plain = max((v for k, v in errs.items() if k.startswith("rel_")), default=0.0)
        key = f"tol {tol:g}"
        w = worst.setdefault(key, [0.0, 0.0, ""])
        if scaled >= w[0]:
            w[0], w[2] = scaled, what
        w[1] = max(w[1], plain)
    for key, (scaled, plain, what) in sorted(worst.items()):
        tr.write_line(f"{key}: worst scaled error {scaled:.3g} ({what}); worst plain relative error {plain:.3g}")
