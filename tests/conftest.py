import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_sessionstart(session):
    # Build libhcr.so in-tree if it is missing or stale (nvcc cross-compiles
    # without a GPU), so the binding can load it.
    import importlib.util
    path = os.path.join(ROOT, "kv_cache_restoration_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("hcr_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running GPU case at full workload size")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when no GPU is present: the product path
    # has no CPU fallback.  Only the marker selects them.
    pass


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU; run it with -m gpu on a GPU machine")
    return torch.device("cuda:0")
