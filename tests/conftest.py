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
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def guarded_outputs(request, monkeypatch):
    """GPU tests: the binding's device allocations (outputs, workspaces) get
    canary guard regions, checked after the test (tests/_util.py)."""
    if "gpu" not in request.keywords:
        yield
        return
    import torch
    if not torch.cuda.is_available():
        yield
        return
    from tests._util import GuardedAlloc, GuardedTorch
    from moe_routed_expert_gb300 import binding
    alloc = GuardedAlloc()
    monkeypatch.setattr(binding, "torch", GuardedTorch(torch, alloc))
    yield alloc
    alloc.check()
