import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_collection_modifyitems(config, items):
    """Runs a test file that sets a module-level RUN_ORDER after the files
    that set none, lowest first (a stable sort: the order within and among
    the other files stays as collected).  Under -x, a failure in such a
    file then comes after every other test has run."""
    items.sort(key=lambda item: getattr(getattr(item, "module", None), "RUN_ORDER", 0))


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def ora():
    import oracle
    return oracle.default()


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
