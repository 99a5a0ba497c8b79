import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size case")
    config.addinivalue_line("markers", "cpu: runs without a GPU")


def read_golden(name):
    """Rows of a golden fixture (comment lines dropped), split on whitespace."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True


def pytest_terminal_summary(terminalreporter):
    """The parity report: every check_errors call of the session (max-normalised error and
    its bound, and the per-element error with a floor of 1e-3 rms(ref))."""
    try:
        from gpu_util import REPORT
    except Exception:
        return
    if not REPORT:
        return
    tr = terminalreporter
    tr.section("parity report")
    tr.write_line(f"{'check':70s} {'out':5s} {'max-norm':>9s} {'bound':>7s} {'elem max':>9s} {'p99.9':>9s} {'median':>9s}")
    for test, kind, rel, tol, emax, ep, emed in REPORT:
        tr.write_line(f"{test[-70:]:70s} {kind:5s} {rel:9.2e} {tol:7.0e} {emax:9.2e} {ep:9.2e} {emed:9.2e}")
