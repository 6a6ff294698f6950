"""Failure detection without a GPU fault.  Every wait inside the library's kernels is bounded;
when one runs out, the kernel records Q2_ERR_TIMEOUT in the workspace status word and returns
instead of hanging.  q2_selftest_wait_timeout makes such a wait run out (a barrier that
nothing completes), and these tests check the status the host reads and that the context
still serves ordinary calls afterwards."""
import time

import numpy as np
import pytest

from _util import check_gemm, to_dev
from speculative_decode_verifier_gb300 import synth

pytestmark = pytest.mark.gpu

Q2_OK, Q2_ERR_TIMEOUT = 0, 6


@pytest.fixture(scope="module")
def env(orc):
    import torch

    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    q2v.load()
    return torch.device("cuda:0"), q2v, orc


def test_bounded_wait_gives_up_and_reports_timeout(env):
    dev, q2v, _ = env
    ws = q2v.workspace(256, dev)
    t0 = time.monotonic()
    q2v.q2_selftest_wait_timeout(ws)
    st = q2v.q2_get_device_status(ws)  # synchronises the stream
    dt = time.monotonic() - t0
    assert st == Q2_ERR_TIMEOUT, q2v.status_string(st)
    assert 0.9 < dt < 30.0, dt         # the wait's limit is one second
    assert q2v.q2_get_device_status(ws) == Q2_OK  # reading cleared the word


def test_context_serves_calls_after_a_timeout(env):
    dev, q2v, orc = env
    ws = q2v.workspace(256, dev)
    q2v.q2_selftest_wait_timeout(ws)
    assert q2v.q2_get_device_status(ws) == Q2_ERR_TIMEOUT
    g = synth.config_gemm(0, M=5, N=512, K=256)
    Y = q2v.q2_tiny_gemm(to_dev(g["W"].reshape(-1), dev), g["N"], g["K"], to_dev(g["A"], dev)).cpu().numpy()
    Yo, absY = orc.gemm(g["W"], g["N"], g["K"], g["A"])
    check_gemm(Y, Yo, absY, "after a timeout")
