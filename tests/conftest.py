import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and libfcomm")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


def pytest_terminal_summary(terminalreporter):
    """The y comparisons of the session: largest error in bf16 ulps and the
    bit-exact fraction, per test and over all of them."""
    try:
        from gpu_util import Y_STATS
    except ImportError:
        return
    if not Y_STATS:
        return
    tr = terminalreporter
    tr.section("y (RMSNorm output) against the oracle, in bf16 ulps of the oracle's value")
    n = sum(s[2] for s in Y_STATS)
    worst = max(s[3] for s in Y_STATS)
    exact = sum(s[2] * s[4] for s in Y_STATS) / n
    tr.write_line(f"{len(Y_STATS)} comparisons, {n} elements: max |dy| = {worst:.3f} ulp, "
                  f"{exact:.6f} of all elements bit-exact, lowest per-comparison bit-exact "
                  f"fraction {min(s[4] for s in Y_STATS):.6f}")
    for test, what, size, mu, ex in Y_STATS:
        tr.write_line(f"  {test} [{what}]: {size} elements, max {mu:.3f} ulp, bit-exact {ex:.6f}")
