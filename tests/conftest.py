import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def page_facts() -> dict:
    """Parse tests/golden/page_facts.txt into {key: number}."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", "page_facts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = float(v) if "." in v else int(v)
    return out


@pytest.fixture(scope="session")
def facts():
    return page_facts()


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle
