"""The multi-GPU path is replicas only: every rank runs the whole step on its own GPU and the job
reports the slowest rank.  These tests run that host logic as two gloo processes on the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        q.put((rank, bench.max_over_ranks(10.0 + 7.5 * rank), bench.max_over_ranks(-1.0 - rank)))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_slowest_replica_is_reported_on_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 17.5, -1.0), (1, 17.5, -1.0)]


def test_single_process_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


@pytest.mark.parametrize("rank,expect_output", [(0, True), (1, False)])
def test_reference_arm_prints_on_rank_zero_only(rank, expect_output):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if expect_output:
        d = json.loads(lines[-1])
        assert d["impl"] == "reference" and d["higher_is_better"] is False and d["value"] > 0
        # the line reports exactly the steps it ran, and the contract's e2e and baseline blocks
        assert d["steps"] == 1 and d["warmup"] == 3
        assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
        cb = d["cpu_baseline"]
        assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
        # the same config, metric and unit as the device arm's line
        sys.path.insert(0, ROOT)
        import bench
        assert d["config"] == bench.run_config(2) and d["metric"] == bench.METRIC and d["unit"] == "µs"
    else:
        assert lines == []
