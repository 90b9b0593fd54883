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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _name_tolerance_records(request):
    """Tag the accuracy records a test makes with its node id."""
    import tolerance
    start = len(tolerance.RECORDS)
    yield
    for r in tolerance.RECORDS[start:]:
        r.setdefault("test", request.node.nodeid)
        r.setdefault("gpu", "gpu" in request.node.keywords)


def pytest_terminal_summary(terminalreporter):
    """Every GPU-vs-oracle comparison of the run: the plain max abs error beside the
    max abs error beyond the bf16 output rounding (the quantity the bar bounds)."""
    import tolerance
    records = [r for r in tolerance.RECORDS if r.get("gpu")]
    if not records:
        return
    tr = terminalreporter
    tr.section("accuracy against the oracle (max abs errors in units of RMS(oracle))")
    tr.write_line(f"{'rel L2':>9} {'plain':>9} {'excess':>9}  test :: output")
    worst = {"rel_l2": 0.0, "plain": 0.0, "excess": 0.0}
    for r in records:
        rms = r["rms"] if r["rms"] > 0 else 1.0
        plain, excess = r["max_abs"] / rms, r["max_abs_excess"] / rms
        worst["rel_l2"] = max(worst["rel_l2"], r["rel_l2"])
        worst["plain"] = max(worst["plain"], plain)
        worst["excess"] = max(worst["excess"], excess)
        tr.write_line(f"{r['rel_l2']:9.2e} {plain:9.2e} {excess:9.2e}  "
                      f"{r.get('test', '?')} :: {r['what']}")
    tr.write_line(f"worst: rel L2 {worst['rel_l2']:.2e} (bar 1e-2), plain max abs "
                  f"{worst['plain']:.2e} RMS, beyond the output rounding {worst['excess']:.2e} "
                  f"RMS (bar 2e-2)")
