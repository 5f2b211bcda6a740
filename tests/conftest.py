import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libar.so")


@pytest.fixture(scope="session")
def orc():
    """The oracle; ORACLE_LIB selects another build of it (the mutation test plants
    mistakes in copies of the oracle and checks that the pins reject each one)."""
    import oracle
    path = os.environ.get("ORACLE_LIB")
    return oracle.Oracle(path) if path else oracle.get()
