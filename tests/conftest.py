import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


@pytest.fixture(scope="session")
def ref():
    """The fp64 oracle.  OSATTN_ORACLE_DIR points the pins at another copy
    of it (used by the planted-mistake test)."""
    alt = os.environ.get("OSATTN_ORACLE_DIR")
    if alt:
        spec = importlib.util.spec_from_file_location(
            "oracle_under_test", os.path.join(alt, "__init__.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    else:
        import oracle as mod
    mod.build()
    return mod
