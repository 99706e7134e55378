import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """key: value lines of a fixture under tests/golden (comments start with #)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """One line with the session's parity totals against the oracle (gpu_util.PARITY), and the
    same as JSON in $SPEC_PARITY_JSON when that is set."""
    try:
        from gpu_util import PARITY
    except ImportError:
        return
    if not (PARITY["proposal_requests"] or PARITY["verify_requests"]):
        return
    terminalreporter.write_line(
        "parity vs oracle: proposals {proposal_exact}/{proposal_requests} requests identical, "
        "{proposal_margin_cases} CDF-margin cases; verify {verify_exact}/{verify_requests} "
        "identical, {verify_margin_cases} margin cases".format(**PARITY))
    path = os.environ.get("SPEC_PARITY_JSON")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(PARITY, f)
