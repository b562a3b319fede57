import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of oracle time)")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) when no GPU is present, so that a
    # plain `pytest tests/` on a CPU-only machine still runs the CPU suite.
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


def read_golden(name):
    """Rows of a golden file: lists of '|'-separated fields, comments dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            rows.append([part.split() for part in line.split("|")])
    return rows


def pytest_terminal_summary(terminalreporter):
    # what each parity comparison left out or held to a looser bound: near-tie
    # pixels (checked at the bound a flipped decision allows), splats left out
    # of a backward comparison, and cancellation-bound gradient elements
    mod = sys.modules.get("gpu_util")
    log = getattr(mod, "PARITY_LOG", None) if mod is not None else None
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity exclusions and near-tie checks")
    for rec in log:
        rest = ", ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}"
                         for k, v in rec.items() if k != "test")
        tr.write_line(f"{rec['test']}: {rest}")
    path = os.environ.get("GS_PARITY_LOG")
    if path:
        import json

        with open(path, "w") as f:
            for rec in log:
                f.write(json.dumps(rec) + "\n")
