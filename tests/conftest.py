import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the hand-written sm_103a kernels)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # The no-allocation entry point's test file is collected last on purpose (see its docstring).
    items.sort(key=lambda it: 1 if os.path.basename(str(it.fspath)).startswith("test_zz_") else 0)


@pytest.fixture(autouse=True)
def _checked_build_records_no_violation(request):
    """Under HS_LIB_VARIANT=checked (the bounds-checked library), every GPU test must also end with no
    bounds violation recorded by any kernel."""
    yield
    if os.environ.get("HS_LIB_VARIANT") == "checked" and request.node.get_closest_marker("gpu"):
        import torch
        if torch.cuda.is_available():
            import sparse_mla_kv_gb300 as hs
            assert hs.check_status() == 0, "a kernel of the bounds-checked build recorded a violation"
