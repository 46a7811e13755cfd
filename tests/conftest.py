import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def _ratio_keys(rec):
    return [k for k in rec if k.endswith("_ratio") or k.startswith("elem_ratio")]


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The worst use of each tolerance the parity comparisons reached in this session."""
    try:
        from parity_util import ACHIEVED
    except Exception:
        return
    if not ACHIEVED:
        return
    worst = {}
    for rec in ACHIEVED:
        for k in _ratio_keys(rec):
            key = (rec["kind"], k)
            if key not in worst or rec[k] > worst[key][0]:
                worst[key] = (rec[k], rec["what"])
    terminalreporter.write_sep("-", f"parity achieved ({len(ACHIEVED)} comparisons): "
                                    "worst measured/bound per tolerance")
    for (kind, k), (v, what) in sorted(worst.items()):
        terminalreporter.write_line(f"{kind:16s} {k:22s} {v:7.3f}  ({what})")
    path = os.environ.get("MHA_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump({"comparisons": ACHIEVED,
                       "worst": {f"{kind}.{k}": {"ratio": v, "what": what}
                                 for (kind, k), (v, what) in sorted(worst.items())}}, f,
                      indent=1)
