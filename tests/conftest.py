import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(scope="session", autouse=True)
def _build_oracle():
    import oracle
    oracle.build()


def pytest_terminal_summary(terminalreporter):
    """Report the achieved parity errors (max|err|/max|ref|) next to their bounds: per test, the
    comparison closest to its bound; all of them go to $M3_PARITY_LOG when that is set."""
    try:
        from parity_util import MARGINS
    except ImportError:
        return
    if not MARGINS:
        return
    worst = {}
    for test, what, err, tol in MARGINS:
        if test not in worst or err / tol > worst[test][1] / worst[test][2]:
            worst[test] = (what, err, tol)
    tr = terminalreporter
    tr.write_sep("-", f"parity margins: {len(MARGINS)} comparisons, closest to its bound per test")
    for test, (what, err, tol) in sorted(worst.items(), key=lambda kv: -kv[1][1] / kv[1][2]):
        tr.write_line(f"{err:9.2e} / {tol:7.0e} = {err / tol:6.3f}  {test}  [{what}]")
    path = os.environ.get("M3_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            for test, what, err, tol in MARGINS:
                f.write(f"{err:.4e}\t{tol:.0e}\t{test}\t{what}\n")
