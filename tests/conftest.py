import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmoe_r3.so")
    config.addinivalue_line("markers", "slow: large sizes")


@pytest.fixture(scope="session")
def oracle():
    from oracle import oracle as O
    O.build()
    return O


# Output errors of the parity tests, printed as a table after the run (the
# per-row bar is asserted by each test; the element-wise error is reported).
_PARITY = []


@pytest.fixture
def parity_report(request):
    """parity_report(what, y, ref): record the per-row and element-wise
    relative errors of y against the oracle's ref (float arrays [rows, cols])."""
    from tests.helpers import elem_rel_err, row_rel_err

    def add(what, y, ref):
        r, e = row_rel_err(y, ref), elem_rel_err(y, ref)
        _PARITY.append((request.node.nodeid.split("::")[-1], what, y.shape[0], float(r.max()), float(e.max()),
                        float(e.mean())))
        return r
    return add


def pytest_terminal_summary(terminalreporter):
    if not _PARITY:
        return
    tr = terminalreporter
    tr.section("parity against the CPU oracle (row: max|y-ref|/max|ref| per row, bar 2e-2; "
               "elem: |y-ref|/max(|ref|, 1e-2 rowmax))")
    for test, what, rows, rmax, emax, emean in _PARITY:
        tr.write_line(f"{test:<48} {what:<28} rows={rows:<7} row_max={rmax:.2e} elem_max={emax:.2e} "
                      f"elem_mean={emean:.2e}")
