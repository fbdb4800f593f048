import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libvbs.so")
    config.addinivalue_line("markers", "slow: long-running (full-size) case")


@pytest.fixture(scope="session")
def golden():
    import json

    def load(name):
        with open(os.path.join(ROOT, "tests", "golden", name)) as f:
            return json.load(f)
    return load


@pytest.fixture(autouse=True)
def _score_error_scope(request):
    """Tag the harness's relative-score-error record with the running test's id."""
    try:
        from tests import harness
    except Exception:            # the harness needs torch; tests that do not are unaffected
        yield
        return
    harness.CURRENT_TEST[0] = request.node.nodeid
    yield
    harness.CURRENT_TEST[0] = "(outside a test)"


def pytest_terminal_summary(terminalreporter):
    """The largest relative score error (|gpu - ref| / |ref|) each beam test saw, worst first."""
    harness = sys.modules.get("tests.harness")
    if harness is None or not harness.REL_ERR:
        return
    rows = sorted(harness.REL_ERR.items(), key=lambda kv: -kv[1][0])
    tr = terminalreporter
    tr.section("relative score error (bound 1e-5)")
    tr.write_line(f"worst over {len(rows)} tests: {rows[0][1][0]:.3e}  ({rows[0][0]}: {rows[0][1][1]})")
    for name, (err, where) in rows:
        tr.write_line(f"{err:.3e}  {name}  [{where}]")
