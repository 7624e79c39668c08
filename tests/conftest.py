import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmla.so")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without a GPU is a configuration error, not a skip, unless
    # the run deselected GPU tests with -m "not gpu".
    pass


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle
