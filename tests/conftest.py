import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")


@pytest.fixture(scope="session", autouse=True)
def _library_under_test():
    """SWIGLU_TEST_DEBUG_LIB=1 runs the whole session on the debug build
    (device index checks).  The binding then waits for every call and raises
    on a device status, so any failed check anywhere fails its test."""
    if os.environ.get("SWIGLU_TEST_DEBUG_LIB") != "1":
        yield
        return
    from backward_tcgen05_tma_gb300 import api, build
    build.build()
    api.use_debug_library(True)
    assert api.lib().swiglu_mlp_debug_build() == 1
    yield
    api.use_debug_library(False)


def device_status(call, ws):
    """The device status that call() leaves in workspace ws: read back with
    swiglu_mlp_query_error, or raised by the binding when it checks every
    call (debug-build sessions)."""
    from backward_tcgen05_tma_gb300 import api
    try:
        call()
    except api.SwigluError as e:
        if e.code in (6, 7):  # SWIGLU_ERR_DEVICE_TIMEOUT, SWIGLU_ERR_DEVICE_BOUNDS
            return e.code
        raise
    return api.swiglu_mlp_query_error(ws)


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def golden_rows(name):
    """Numeric rows of a whitespace-separated fixture under tests/golden/."""
    path = os.path.join(ROOT, "tests", "golden", name)
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([float(t) for t in line.split()])
    return rows
