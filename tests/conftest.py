import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


import json

import pytest


@pytest.fixture(autouse=True)
def _name_parity_records(request):
    import gpu_helpers
    gpu_helpers.CURRENT_TEST[0] = request.node.nodeid
    yield


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("GDN_PARITY_LOG")
    if not path:
        return
    import gpu_helpers
    if not gpu_helpers.RECORDS:
        return
    with open(path, "w") as f:
        for r in gpu_helpers.RECORDS:
            f.write(json.dumps(r) + "\n")
