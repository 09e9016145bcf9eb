import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """With GNN_PARITY_REPORT set, write every GPU comparison's accounting
    (elements, elements passing only through the float32 summation term,
    worst strict ratio), aggregated by what was compared."""
    path = os.environ.get("GNN_PARITY_REPORT")
    mod = sys.modules.get("gpu_util")
    if not path or mod is None:
        return
    import json
    agg = {}
    for r in mod.REPORT:
        a = agg.setdefault(r["what"], {"n": 0, "mag_only": 0, "kink_only": 0,
                                       "kink_elements": 0, "worst_strict_ratio": 0.0,
                                       "comparisons": 0})
        a["n"] += r["n"]
        a["mag_only"] += r["mag_only"]
        a["kink_only"] += r["kink_only"]
        a["kink_elements"] += r["kink_elements"]
        a["worst_strict_ratio"] = max(a["worst_strict_ratio"], r["worst_strict_ratio"])
        a["comparisons"] += 1
    with open(path, "w") as f:
        json.dump(agg, f, indent=1, sort_keys=True)
