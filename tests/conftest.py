import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity cases")


@pytest.fixture(scope="session")
def ref():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _name_error_stats(request):
    from tests import helpers
    helpers.CURRENT_TEST[0] = request.node.nodeid
    yield


def pytest_terminal_summary(terminalreporter):
    from tests import helpers
    if not helpers.ERRSTATS:
        return
    tr = terminalreporter
    tr.section("output error against the oracle (tolerance max 2e-2, mean 2e-3)")
    for name, mx, mean, n in helpers.ERRSTATS:
        tr.write_line("%-90s max|err| %.3e  mean|err| %.3e  (%d values)" % (name, mx, mean, n))
