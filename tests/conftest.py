import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    # libpa.so rebuilt before collection when any source is newer (a no-op otherwise), so a test
    # module that imports the binding at its top never loads a library older than the sources
    _build_and_import(import_binding=False)


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def _build_and_import(import_binding=True):
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "pa_build", os.path.join(ROOT, "paged_kv_cache_bs_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    if not import_binding:
        return None
    import paged_kv_cache_bs_gb300
    return paged_kv_cache_bs_gb300


@pytest.fixture(scope="session")
def pa_host():
    """The binding for host-only calls (argument checks, the page directory): no GPU needed."""
    return _build_and_import()


@pytest.fixture(scope="session")
def pa():
    """The CUDA library's binding, built in-tree first.  GPU tests need a GPU:
    there is no fallback, so a missing device is an error, not a skip."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "pa_build", os.path.join(ROOT, "paged_kv_cache_bs_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import paged_kv_cache_bs_gb300
    return paged_kv_cache_bs_gb300
