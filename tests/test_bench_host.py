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
    assert rec["kernel"].startswith("moe_stream_kernel<1,1>")
    assert int(rec["bytes"]) > 0 and int(rec["units"]) > 0 and rec["unit"] == "active_experts"
    assert re.fullmatch(r"[0-9a-f]{16}", rec["sources"])
    assert re.fullmatch(r"[0-9a-f]{16}", bench._kernel_source_digest())
