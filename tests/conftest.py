import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _name_parity_comparisons(request):
    """Tag the parity margins recorded by pkv_testutil with the running test."""
    try:
        import pkv_testutil
    except Exception:  # pragma: no cover - helper not importable
        yield
        return
    pkv_testutil.CURRENT_TEST["id"] = request.node.nodeid
    yield


def pytest_terminal_summary(terminalreporter):
    """Print the parity margins: worst |gpu - oracle| / tolerance bound per test."""
    mod = sys.modules.get("pkv_testutil")
    margins = getattr(mod, "MARGINS", None) if mod else None
    if not margins:
        return
    worst = {}
    for m in margins:
        key = m["test"]
        if key not in worst or m["ratio"] > worst[key]["ratio"]:
            worst[key] = m
    rows = sorted(worst.values(), key=lambda m: -m["ratio"])
    tr = terminalreporter
    tr.write_sep("-", "parity margins: worst |gpu - oracle| / (1e-2 * max(1, |oracle|)) per test")
    for m in rows:
        name = m["test"].split("::", 1)[-1]
        tr.write_line(f"{m['ratio']:6.3f}  max|err| {m['max_err']:.2e}  "
                      f"{m['elements']:>10d} elems  {name}  [{m['what']}]")
    fams = {}
    for m in rows:
        fam = m["test"].split("::")[0].rsplit("/", 1)[-1]
        fams[fam] = max(fams.get(fam, 0.0), m["ratio"])
    tr.write_line("worst per file: " + ", ".join(f"{k} {v:.3f}" for k, v in sorted(fams.items())))
