import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs an sm_103a GPU (GB300); runs the CUDA path")


def pytest_collection_modifyitems(config, items):
    # keep the no-GPU tests green on a box without CUDA: a gpu test that is
    # selected there fails loudly instead of silently skipping.
    pass


def pytest_terminal_summary(terminalreporter):
    """How much of the parity bounds the GPU results used (largest shares)."""
    gc = sys.modules.get("gpu_common")
    rows = getattr(gc, "MARGINS", None) if gc is not None else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("parity margins (share of the bound used; largest first)")
    worst_o = max(r[2] for r in rows)
    lse = [r for r in rows if r[4] is not None]
    worst_l = max((r[4] for r in lse), default=0.0)
    tr.write_line(f"{len(rows)} comparisons; largest share of the O bound {worst_o:.3f}, "
                  f"of the LSE bound {worst_l:.3f}")
    for r in sorted(rows, key=lambda r: -r[2])[:8]:
        lpart = f", max|dLSE| {r[3]:.2e} ({r[4]:.3f})" if r[3] is not None else ""
        tr.write_line(f"  {r[0]}: max|dO| {r[1]:.2e} ({r[2]:.3f}){lpart}")
