import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libvst")


def load_page_constants():
    path = os.path.join(ROOT, "tests", "golden", "page_constants.txt")
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, _, cite = line.partition("|")
            name, value = head.split()
            assert cite.strip(), "constant %s has no citation" % name
            out[name] = int(value)
    return out


@pytest.fixture(scope="session")
def page_constants():
    return load_page_constants()
