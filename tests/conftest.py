import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_sessionstart(session):
    # Build libskinny.so (nvcc, sm_103a) and the oracle (gcc) if they are
    # missing or older than their sources; both builds are incremental.
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "_skinny_build", os.path.join(ROOT, "fp8_weight_only_skinny_gb300", "build.py"))
    skbuild = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(skbuild)   # without importing the package (it loads the .so)
    skbuild.build()
    import oracle

    oracle.build()
