import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per-workload parity tallies (rows compared, near-threshold counts, worst
    deviations) of the comparisons this session ran; also written as JSON to
    the path in RLK_PARITY_REPORT when that is set."""
    mod = sys.modules.get("_oracle_check")
    if mod is None or not mod.REPORT:
        return
    import json
    terminalreporter.section("parity summary (GPU against the oracle)")
    for name, d in mod.REPORT.items():
        terminalreporter.write_line(f"{name}: " + json.dumps(d, sort_keys=True))
    path = os.environ.get("RLK_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(mod.REPORT, f, indent=1, sort_keys=True)


def pytest_sessionfinish(session, exitstatus):
    mod = sys.modules.get("_oracle_check")
    if mod is not None:
        mod.shutdown()
