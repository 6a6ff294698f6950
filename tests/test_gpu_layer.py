"""The verifier-layer chain on the GPU against the fp64 oracle: the Q, K, V and O projections
(4096 x 4096 Q2B32 linears at M=5) and the routed MoE FFN (64 experts, H=4096, F=2048, top-6)
enqueued back to back on one stream, each kernel launched with programmatic dependent launch
so that a GEMM's weight loads go out before the previous kernel has finished, then pq_verify
(S=3, k=4, V=129,280) as the verifier step ends.  Run eagerly and replayed from one CUDA
graph; every output is held to the oracle under the usual rules."""
import numpy as np
import pytest

from _util import check_gemm, compare_verify, to_dev
from speculative_decode_verifier_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer(orc):
    import torch

    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    q2v.load()
    dev = torch.device("cuda:0")
    g = synth.config_gemm(1)
    N, K, M = g["N"], g["K"], g["M"]
    Ws = [synth.q2b32_weights(synth.Streams(9000 + i), N, K) for i in range(4)]
    m = synth.config_moe(2)
    v = synth.config_verify(3)
    want = dict(lin=[orc.gemm(W, N, K, g["A"]) for W in Ws],
                moe=orc.moe(m["Wg"], m["Wu"], m["Wd"], m["E"], m["H"], m["F"], m["topk"], m["X"], m["router"]),
                pq=orc.pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], v["T"],
                                 want_probs=True))
    d = dict(W=[to_dev(W.reshape(-1), dev) for W in Ws], A=to_dev(g["A"], dev),
             Wg=to_dev(m["Wg"].reshape(-1), dev), Wu=to_dev(m["Wu"].reshape(-1), dev),
             Wd=to_dev(m["Wd"].reshape(-1), dev), X=to_dev(m["X"], dev), R=to_dev(m["router"], dev),
             **{n: to_dev(v[n], dev) for n in ("target", "draft", "drafts", "u_acc", "u_fin")})
    out = dict(Y=[torch.full((M, N), float("nan"), device=dev) for _ in range(4)],
               Ym=torch.full((M, m["H"]), float("nan"), device=dev),
               n=torch.full((v["target"].shape[0],), -7, dtype=torch.int32, device=dev),
               t=torch.full(v["target"].shape[:2], -7, dtype=torch.int32, device=dev))
    ws = dict(lin=q2v.workspace(q2v.q2_tiny_gemm_workspace(M, N, K), dev),
              moe=q2v.workspace(q2v.q2_moe_grouped_workspace(M, m["E"], m["topk"], m["H"], m["F"]), dev),
              pq=q2v.workspace(q2v.pq_verify_workspace(*v["target"].shape[:1], v["target"].shape[1] - 1,
                                                       v["target"].shape[2]), dev))

    def run():
        # one workspace shared by the four projections, as a layer would run them
        for i in range(4):
            q2v.q2_tiny_gemm(d["W"][i], N, K, d["A"], Y=out["Y"][i], ws=ws["lin"])
        q2v.q2_moe_grouped(d["Wg"], d["Wu"], d["Wd"], m["E"], m["H"], m["F"], m["topk"], d["X"], d["R"],
                           Y=out["Ym"], ws=ws["moe"])
        q2v.pq_verify(d["target"], d["draft"], d["drafts"], d["u_acc"], d["u_fin"], v["T"], n_acc=out["n"],
                      tokens=out["t"], ws=ws["pq"])

    return dict(q2v=q2v, dev=dev, run=run, out=out, want=want, ws=ws, v=v)


def _check_outputs(L):
    import torch
    torch.cuda.synchronize()
    for w in L["ws"].values():
        assert L["q2v"].q2_get_device_status(w) == 0
    for i in range(4):
        Yo, absY = L["want"]["lin"][i]
        check_gemm(L["out"]["Y"][i].cpu().numpy(), Yo, absY, f"projection {i}")
    mo = L["want"]["moe"]
    err = np.abs(L["out"]["Ym"].cpu().numpy().astype(np.float64) - mo["Y"])
    assert np.all(err <= mo["tol"]), f"MoE: worst err/tol {np.max(err / mo['tol'])}"
    v = L["v"]
    stats = compare_verify(L["out"]["n"].cpu().numpy(), L["out"]["t"].cpu().numpy(), L["want"]["pq"], v["u_acc"],
                           v["u_fin"], v["target"].shape[1] - 1)
    assert stats["exact"] + stats["mismatches_at_near_ties"] == stats["sessions"]


def _poison(L):
    for Y in L["out"]["Y"]:
        Y.fill_(float("nan"))
    L["out"]["Ym"].fill_(float("nan"))
    L["out"]["n"].fill_(-7)
    L["out"]["t"].fill_(-7)


def test_layer_chain_eager(layer):
    _poison(layer)
    layer["run"]()
    _check_outputs(layer)


def test_layer_chain_graph_replays(layer):
    import torch
    layer["run"]()  # warm-up outside capture (device attributes are cached on the first call)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        layer["run"]()
    for _ in range(2):  # the second replay reuses every workspace the first one left behind
        _poison(layer)
        torch.cuda.synchronize()
        gr.replay()
        _check_outputs(layer)
