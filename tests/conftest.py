import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libqz.so")
    # build the library and the oracle once (in-tree, incremental) before collection
    import __graft_entry__
    __graft_entry__.build()


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def golden_path(name: str) -> str:
    return os.path.join(ROOT, "tests", "golden", name)


def read_golden(name: str):
    """Rows of whitespace-separated fields of a golden file, comments dropped."""
    rows = []
    with open(golden_path(name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Report how many GEMM output elements passed only because of the half-bf16-ulp
    term of the tolerance (the rest are within 1e-3 * sum |a*b| alone)."""
    try:
        from gpu_util import HALF_ULP_TALLY
    except Exception:  # pragma: no cover
        return
    if not HALF_ULP_TALLY:
        return
    total = sum(n for _, n, _ in HALF_ULP_TALLY)
    extra = sum(h for _, _, h in HALF_ULP_TALLY)
    terminalreporter.write_sep("-", "GEMM tolerance audit")
    terminalreporter.write_line(f"{len(HALF_ULP_TALLY)} GEMM checks, {total} elements; {extra} pass only through "
                                f"the half-bf16-ulp term of the tolerance")
    for what, n, h in HALF_ULP_TALLY:
        if h:
            terminalreporter.write_line(f"  {what}: {h} of {n}")
