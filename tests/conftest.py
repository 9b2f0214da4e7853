import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


# Run last, whatever the file order: the tests of the decode entry point that
# keeps its scratch in a library-owned device array.
LAST = "test_zz_no_alloc.py"


def pytest_collection_modifyitems(session, config, items):
    items.sort(key=lambda it: os.path.basename(str(it.fspath)) == LAST)


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


@pytest.fixture(scope="session")
def pkv():
    """The built CUDA library's binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_268_gb300 import _binding, build
    build.build()
    _binding.load_library()
    return _binding
