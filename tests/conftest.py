import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


def pytest_sessionfinish(session, exitstatus):
    """With FA_ERROR_LOG set, write the errors every parity comparison measured (JSON lines)."""
    path = os.environ.get("FA_ERROR_LOG")
    mod = sys.modules.get("gpu_util")
    if not path or mod is None:
        return
    import json
    with open(path, "w") as f:
        for rec in mod.ERROR_LOG:
            f.write(json.dumps(rec) + "\n")
