import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


@pytest.fixture(scope="session")
def golden():
    import json

    with open(os.path.join(ROOT, "tests", "golden", "worked_numbers.json")) as f:
        return json.load(f)


def build_native():
    """Build libpkv.so if stale, without importing the package first."""
    import importlib.util

    path = os.path.join(ROOT, "paged_kv_cache_49_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("pkv_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()
