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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmbglu.so")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


@pytest.fixture(autouse=True)
def _parity_label(request):
    import tolerance
    tolerance.CURRENT_TEST[0] = request.node.nodeid
    yield


def pytest_sessionfinish(session, exitstatus):
    """Writes every parity comparison of the session (label, statistics,
    verdict) as JSON to $MBGLU_PARITY_STATS, by default parity_stats.json in
    the repository's untracked output folder."""
    import json
    import tolerance
    if not tolerance.RECORDS:
        return
    path = os.environ.get("MBGLU_PARITY_STATS", os.path.join(ROOT, "gpurun_out", "parity_stats.json"))
    try:
        os.makedirs(os.path.dirname(path), exist_ok=True)
        with open(path, "w") as f:
            json.dump(tolerance.RECORDS, f, indent=0)
    except OSError:
        pass
