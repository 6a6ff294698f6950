import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def orc():
    from oracle import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Near-tie report: per test, the verify sessions compared with the oracle, how many matched
    exactly, how many had a uniform within 1e-5 of an accept ratio or of a draw's CDF cell edge,
    and how many of those near-ties gave a different (still admissible) result."""
    util = sys.modules.get("_util")
    log = getattr(util, "NEAR_TIE_LOG", None)
    if not log:
        return
    keys = ("sessions", "exact", "accept_near_ties", "draw_near_ties", "mismatches_at_near_ties")
    per = {}
    for test, st in log:
        acc = per.setdefault(test, dict.fromkeys(keys, 0))
        for k in keys:
            acc[k] += int(st.get(k, 0))
    tr = terminalreporter
    tr.write_sep("-", "near-tie report (verify sessions vs the oracle)")
    tr.write_line("test | " + " | ".join(keys))
    for test, acc in per.items():
        tr.write_line(f"{test} | " + " | ".join(str(acc[k]) for k in keys))
    out = os.environ.get("Q2V_NEAR_TIE_REPORT")
    if out:
        import json
        with open(out, "w") as f:
            json.dump(per, f, indent=1)
