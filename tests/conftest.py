import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test (excluded from the default CPU run)")


def pytest_collection_modifyitems(config, items):
    # slow CPU tests run only when asked for with -m slow
    markexpr = config.getoption("-m") or ""
    if "slow" in markexpr:
        return
    skip = pytest.mark.skip(reason="slow: run with -m slow")
    for item in items:
        if "slow" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """The output checks' unmodified error figures and how many elements each
    widening of the 1e-2 * rms(Y) bound admitted (tests/gpu_util.py)."""
    mod = sys.modules.get("gpu_util")
    log = getattr(mod, "TOLERANCE_LOG", None) if mod else None
    if not log:
        return
    tr = terminalreporter
    tr.section("output tolerance book-keeping")
    tr.write_line(f"{'check':44s} {'elements':>10s} {'rel_fro':>9s} {'max|err|/rms':>12s} "
                  f"{'>1e-2rms':>9s} {'>+ulp/2':>8s}")
    for r in log:
        tr.write_line(f"{r['what'][:44]:44s} {r['elements']:10d} {r['rel_fro']:9.2e} "
                      f"{r['max_abs_over_rms']:12.4f} {r['needed_half_ulp']:9d} "
                      f"{r['needed_lora_slack']:8d}")
