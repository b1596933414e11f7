import os
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_sessionfinish(session, exitstatus):
    """Write the parity records of this session (tests/parity.py AUDIT) as JSON: to
    $HRA_PARITY_AUDIT, else parity_audit.json in the system's temporary directory."""
    try:
        import parity
    except Exception:
        return
    if not parity.AUDIT:
        return
    import json
    path = os.environ.get("HRA_PARITY_AUDIT") or os.path.join(tempfile.gettempdir(), "parity_audit.json")
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "w") as f:
        json.dump(parity.AUDIT, f, indent=0)
