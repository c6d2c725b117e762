import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Both pass rates of the floating-point comparisons: every element met the relaxed
    bound max(1e-2, 1 bf16 ulp) (the tests assert it); how many also met the literal
    max-abs 1e-2, overall and for the comparisons where some did not."""
    try:
        import tol
    except ImportError:
        return
    if not tol.STATS:
        return
    n = sum(s[1] for s in tol.STATS)
    lit = sum(s[2] for s in tol.STATS)
    tr = terminalreporter
    tr.section("tolerance pass rates (bf16 outputs against the fp64 oracle)")
    tr.write_line(f"{len(tol.STATS)} comparisons, {n} elements: relaxed bound max(1e-2, 1 ulp) "
                  f"met by all that passed; literal max-abs 1e-2 met by {lit} "
                  f"({100.0 * lit / n:.4f} %)")
    short = sorted((s for s in tol.STATS if s[2] < s[1]), key=lambda s: s[2] / s[1])
    for what, m, k, worst in short[:12]:
        tr.write_line(f"  {what}: {m - k} of {m} elements beyond 1e-2 (worst {worst:.3g})")
    if len(short) > 12:
        tr.write_line(f"  ... and {len(short) - 12} more comparisons with elements beyond 1e-2")
