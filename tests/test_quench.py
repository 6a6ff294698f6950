"""The host-side yield-quench controller ("ds4-on-spark" README, "The break-even law"): per
verify step the regret grows by guard - (n_accepted + 1), and a session is quenched for good
once it exceeds the threshold.  Expected values are worked out by hand from that rule."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def q2v():
    from speculative_decode_verifier_gb300 import build, q2v as mod
    build.build()
    mod.load()
    return mod


def test_one_token_per_step_quenches_on_the_fourth_step(q2v):
    # guard 2.16, 1 token per step: regret 1.16, 2.32, 3.48 (<= 4), 4.64 (> 4) -> quenched at step 4
    qc = q2v.YieldQuench(1)
    got = [qc.update([0]) for _ in range(4)]
    assert got == [0, 0, 0, 1] and qc.quenched() == [True]
    assert abs(qc.regret()[0] - 4 * 1.16) < 1e-12
    assert qc.update([0]) == 0 and abs(qc.regret()[0] - 4 * 1.16) < 1e-12  # terminal: no more accounting


def test_threshold_is_strict(q2v):
    # guard 2, 1 token per step: regret exactly 4.0 after 4 steps does not quench, 5.0 does
    qc = q2v.YieldQuench(1, guard=2.0, threshold=4.0)
    assert [qc.update([0]) for _ in range(5)] == [0, 0, 0, 0, 1]


def test_winning_requests_never_quench_and_bank_credit(q2v):
    qc = q2v.YieldQuench(2)
    for _ in range(50):
        assert qc.update([4, 2]) == 0  # 5 and 3 tokens per step: both above the break-even
    assert qc.quenched() == [False, False]
    assert abs(qc.regret()[0] - 50 * (2.16 - 5)) < 1e-9 and abs(qc.regret()[1] - 50 * (2.16 - 3)) < 1e-9
    # credit earned is spent before a deficit can quench: 50 * 0.84 = 42 of credit, then 1 token/step
    steps = 0
    while not qc.quenched()[1]:
        qc.update([4, 0])
        steps += 1
    assert steps == int(np.floor((50 * 0.84 + 4.0) / 1.16)) + 1


def test_sessions_are_independent_and_bad_steps_are_skipped(q2v):
    qc = q2v.YieldQuench(3)
    for _ in range(4):
        qc.update([0, -1, 4])
    assert qc.quenched() == [True, False, False]
    assert qc.regret()[1] == 0.0 and qc.state[1].steps == 0 and qc.state[0].steps == 4


def test_invalid_arguments(q2v):
    import ctypes
    lib = q2v.load()
    assert lib.q2_quench_init(None, 3) == 1
    st = (q2v.QuenchState * 2)()
    assert lib.q2_quench_init(st, 0) == 1
    arr = (ctypes.c_int32 * 2)(0, 0)
    assert lib.q2_quench_update(st, 2, arr, float("nan"), 4.0) == -1
    assert lib.q2_quench_update(st, 2, None, 2.16, 4.0) == -1
