"""Host-side pieces of bench.py that need no GPU: the launch count matches the step's kernels,
and the recorded DRAM-traffic line that the roofline reports parses into the fields bench.py
reads."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_launches_per_step():
    # prep + GEMM; route with X prep, gate/up, prep h, down, combine; statistics + draw
    assert bench.LAUNCHES_PER_STEP == 9


def test_traffic_record_parses():
    rec = bench._traffic_record()
    assert rec is not None
    assert rec["kernel"] == "moe_gateup_stream_kernel"
    assert int(rec["bytes"]) > 0 and int(rec["units"]) > 0 and rec["unit"] == "active_experts"
    assert re.fullmatch(r"[0-9a-f]{16}", rec["sources"])
    assert re.fullmatch(r"[0-9a-f]{16}", bench._kernel_source_digest())


def test_near_tie_counter():
    import numpy as np
    o = dict(n_acc=np.array([1, 2, 0]), tokens=np.array([[5, 9, -1], [5, 6, 7], [3, -1, -1]]),
             ratio=np.array([[0.9, 0.3], [0.9, 0.8], [0.2500001, 0.5]]),
             cell_lo=np.array([0.1, 0.2, 0.3]), cell_hi=np.array([0.2, 0.3, 0.4]))
    u_acc = np.array([[0.5, 0.6], [0.1, 0.1], [0.25, 0.1]], np.float32)
    u_fin = np.array([0.15, 0.299995, 0.35], np.float32)
    n = np.array([1, 2, 1])
    t = np.array([[5, 9, -1], [5, 6, 8], [3, 4, -1]])
    st = bench._near_ties(n, t, o, u_acc, u_fin, 2)
    # session 0 exact; session 1 differs at a draw near-tie (u_fin 1e-5 from the cell edge);
    # session 2 differs at an accept near-tie (u_acc 1e-7 from p/q)
    assert st == dict(sessions=3, exact=1, accept_near_ties=1, draw_near_ties=1, mismatches_at_near_ties=2,
                      mismatches_without_near_tie=0)
    t[0, 1] = 8
    assert bench._near_ties(n, t, o, u_acc, u_fin, 2)["mismatches_without_near_tie"] == 1


def test_timed_traffic_record_parses():
    rec = bench._traffic_record("traffic-timed")
    assert rec is not None and rec["unit"] == "active_experts"
    assert rec["sources"] == bench._traffic_record()["sources"]
    # the timed launches read what the weights need, give or take the L2's write-backs
    assert 6_291_456 <= int(rec["bytes"]) / int(rec["units"]) < 1.1 * 6_291_456
