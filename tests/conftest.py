import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def load_build_module():
    """The library's standalone build script, loaded by path."""
    import importlib.util

    path = os.path.join(ROOT, "combine_get_layout_gb300", "build_lib.py")
    spec = importlib.util.spec_from_file_location("ep_build_lib", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Parse a golden fixture: '#' lines are comments/citations; every other
    line is 'key tok tok ...'.  Returns a list of (key, [tokens])."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            rows.append((key, rest))
    return rows


@pytest.fixture(scope="session")
def golden():
    return read_golden
