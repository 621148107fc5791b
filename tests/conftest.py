import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        with open(os.path.join(GOLDEN, name)) as f:
            return json.load(f)

    return load


def pytest_sessionfinish(session, exitstatus):
    """With GBATTN_GRAD_LOG set, write the measured gradient-error margins of
    every backward comparison of the session to that file (JSON)."""
    path = os.environ.get("GBATTN_GRAD_LOG")
    if not path:
        return
    try:
        from tests.parity_util import GRAD_LOG
    except ImportError:
        return
    import json

    with open(path, "w") as f:
        json.dump(GRAD_LOG, f, indent=0)
