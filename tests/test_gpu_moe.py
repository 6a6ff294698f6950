"""q2_moe_grouped on the GPU against the fp64 oracle: routing ids identical, gate weights to
fp32 rounding, outputs within the propagated bound (2e-3 relative on each contraction plus
the first-order effect of the gate/up tolerance through silu and the down projection)."""
import numpy as np
import pytest

from _util import to_dev
from speculative_decode_verifier_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(orc):
    import torch

    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    q2v.load()
    return torch.device("cuda:0"), q2v, orc


def _run(env, m, renorm=False, ws=None):
    import torch
    dev, q2v, orc = env
    M, topk = m["M"], m["topk"]
    ids = torch.empty((M, topk), dtype=torch.int32, device=dev)
    gw = torch.empty((M, topk), dtype=torch.float32, device=dev)
    Y = q2v.q2_moe_grouped(to_dev(m["Wg"].reshape(-1), dev), to_dev(m["Wu"].reshape(-1), dev),
                           to_dev(m["Wd"].reshape(-1), dev), m["E"], m["H"], m["F"], topk,
                           to_dev(m["X"], dev), to_dev(m["router"], dev), ids_out=ids, w_out=gw,
                           renormalize=renorm, ws=ws)
    o = orc.moe(m["Wg"], m["Wu"], m["Wd"], m["E"], m["H"], m["F"], topk, m["X"], m["router"], renorm=renorm)
    Yg = Y.cpu().numpy().astype(np.float64)
    assert np.array_equal(ids.cpu().numpy(), o["ids"])
    np.testing.assert_allclose(gw.cpu().numpy(), o["weights"], rtol=2e-6, atol=1e-9)
    err = np.abs(Yg - o["Y"])
    assert np.all(err <= o["tol"]), f"worst err/tol {np.max(err / o['tol'])}"
    return Yg, o


def test_moe_config_full_size(env):
    m = synth.config_moe(2)
    Y, o = _run(env, m)
    active = np.unique(o["ids"]).size
    assert 15 <= active <= 30  # ~25 of 64 experts expected for 5 rows x top-6


@pytest.mark.parametrize("over", [
    dict(E=4, H=64, F=96, M=3, topk=2),
    dict(E=8, H=96, F=160, M=5, topk=3),      # odd block counts on both GEMMs
    dict(E=8, H=256, F=128, M=64, topk=2),     # many rows per expert: several slices
    dict(E=256, H=128, F=64, M=4, topk=16),    # the largest E and top-k
    dict(E=16, H=8192, F=256, M=2, topk=4),    # the largest H
    dict(E=64, H=4096, F=2048, M=1, topk=6),   # one row: every active expert has a single column
    dict(E=32, H=1024, F=96, M=8, topk=4),     # all 8 X rows in one MMA column set
    dict(E=256, H=2816, F=160, M=7, topk=16),  # 11 K tiles, the largest E and top-k
    dict(E=8, H=4352, F=64, M=3, topk=2),      # 17 K tiles: 8 splits of 3 would leave 2 empty, so 6 are used
    dict(E=1, H=256, F=128, M=5, topk=1),      # one expert: every row routed to it with gate weight 1
    dict(E=2, H=512, F=256, M=8, topk=2),      # top-k = E: every row routed to every expert
    dict(E=64, H=4096, F=2048, M=8, topk=6),   # 8 rows at full size: up to 48 active experts
    dict(E=64, H=768, F=1024, M=8, topk=8),    # streaming gate+up over 3-tile units (cuts on single tiles)
    dict(E=64, H=256, F=2048, M=7, topk=8),    # streaming gate+up at 7 rows (masked MMA columns)
    dict(E=64, H=256, F=4096, M=3, topk=6),    # streaming gate+up at 3 rows
    dict(E=64, H=8192, F=256, M=3, topk=6),    # streaming down at 3 rows (windows of up to 6 pairs)
    dict(E=64, H=1024, F=256, M=7, topk=8),    # streaming down at 7 rows (windows of up to 14 pairs)
])
def test_shapes(env, over):
    m = synth.config_moe(2, salt=sum(over.values()), **over)
    _run(env, m)


def test_renormalized_gates(env):
    m = synth.config_moe(2, salt=3, E=16, H=256, F=128, M=5, topk=4)
    _run(env, m, renorm=True)


def test_router_ties_go_to_lower_index(env):
    m = synth.config_moe(2, salt=4, E=8, H=64, F=64, M=4, topk=3)
    m["router"][:, :] = 0.0
    m["router"][1, 5] = 1.0
    _run(env, m)


def test_workspace_reuse(env):
    dev, q2v, _ = env
    m = synth.config_moe(2, salt=5, E=8, H=256, F=128, M=5, topk=2)
    ws = q2v.workspace(q2v.q2_moe_grouped_workspace(5, 8, 2, 256, 128), dev)
    a, _ = _run(env, m, ws=ws)
    b, _ = _run(env, m, ws=ws)
    assert np.array_equal(a, b)


def test_verifier_shape_is_deterministic(env):
    # every sum (K tiles, K splits, slots) runs in a fixed order
    m = synth.config_moe(2, salt=6, E=64, H=4096, F=2048, M=5, topk=6)
    a, _ = _run(env, m)
    b, _ = _run(env, m)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("mat", ["Wg", "Wd"])
def test_scale_out_of_range_sets_status(env, mat):
    """A gate (or down) scale of 64 in every expert: the streaming gate+up (or down) kernel, which
    this shape takes, flags Q2_ERR_RANGE in the status word."""
    import torch
    dev, q2v, _ = env
    m = synth.config_moe(2, salt=5, E=8, H=256, F=256, M=5, topk=3)
    W = {k: np.array(m[k], copy=True) for k in ("Wg", "Wu", "Wd")}
    d = W[mat].reshape(-1, W[mat].shape[-2], 12)[:, 0, 8:10]   # block 0 of every row: the d half
    d[:] = synth.fp16_bits(np.full(1, 64.0)).view(np.uint8)
    ws = q2v.workspace(q2v.q2_moe_grouped_workspace(m["M"], m["E"], m["topk"], m["H"], m["F"]), dev)
    q2v.q2_moe_grouped(to_dev(W["Wg"].reshape(-1), dev), to_dev(W["Wu"].reshape(-1), dev),
                       to_dev(W["Wd"].reshape(-1), dev), m["E"], m["H"], m["F"], m["topk"],
                       to_dev(m["X"], dev), to_dev(m["router"], dev), ws=ws)
    torch.cuda.synchronize()
    assert q2v.q2_get_device_status(ws) == 8  # Q2_ERR_RANGE
