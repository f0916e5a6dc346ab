import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the parity tests proper)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    return oracle.load()


@pytest.fixture(scope="session")
def lib():
    """The GPU library's Python binding, built in-tree when missing."""
    from exact_full_reference_gb300 import build as vbuild

    vbuild.build_library()
    import exact_full_reference_gb300 as vqx

    return vqx
