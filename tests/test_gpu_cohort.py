"""The cohort verify at full size: 12 sessions x 5 rows = M=60 against a Q2B32 lm_head
(K=4096, N=129280), then pq_verify (S=12, k=4, V=129280) over the logits -- the launch
configuration the benchmark times."""
import numpy as np
import pytest

from _util import check_gemm, compare_verify, to_dev
from speculative_decode_verifier_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cohort(orc):
    import torch

    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    q2v.load()
    dev = torch.device("cuda:0")
    cfg = synth.CONFIGS[4]
    g = synth.config_gemm(4)
    Yo, absY = orc.gemm(g["W"], g["N"], g["K"], g["A"])
    st = synth.streams(4, salt=1)
    v = synth.verify_inputs(st, cfg["S"], cfg["k"], cfg["V"], 0.0, cfg["noise_std"], cfg["T"],
                            target=Yo.astype(np.float32))
    return dict(dev=dev, q2v=q2v, orc=orc, g=g, Yo=Yo, absY=absY, v=v)


def test_lm_head_gemm_m60_all_outputs(cohort):
    c = cohort
    q2v, dev, g = c["q2v"], c["dev"], c["g"]
    Y = q2v.q2_tiny_gemm(to_dev(g["W"].reshape(-1), dev), g["N"], g["K"], to_dev(g["A"], dev))
    check_gemm(Y.cpu().numpy(), c["Yo"], c["absY"], "cfg4 lm_head")


def test_pq_verify_on_oracle_logits(cohort):
    c = cohort
    q2v, dev, v, orc = c["q2v"], c["dev"], c["v"], c["orc"]
    import torch
    t = {n: to_dev(v[n], dev) for n in ("target", "draft", "drafts", "u_acc", "u_fin")}
    S, k1, V = v["target"].shape
    probs = torch.empty((S, 2 * k1 - 1, V), dtype=torch.float32, device=dev)
    n, toks = q2v.pq_verify(t["target"], t["draft"], t["drafts"], t["u_acc"], t["u_fin"], v["T"], probs=probs)
    o = orc.pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], v["T"], want_probs=True)
    assert np.abs(probs.cpu().numpy().astype(np.float64) - o["probs"]).max() <= 1e-5
    stats = compare_verify(n.cpu().numpy(), toks.cpu().numpy(), o, v["u_acc"], v["u_fin"], k1 - 1)
    assert stats["exact"] + stats["mismatches_at_near_ties"] == S


def test_chained_gemm_then_verify(cohort):
    """GEMM output fed straight into pq_verify on one stream, as the benchmark step runs it.
    The logits differ from the oracle's by the GEMM rounding, so the tokens are held to the
    structural rules and to agreement with the oracle run on the oracle's own logits for
    every session whose decisions are not within 1e-3 of a boundary."""
    c = cohort
    q2v, dev, g, v, orc = c["q2v"], c["dev"], c["g"], c["v"], c["orc"]
    S, k1, V = v["target"].shape
    Y = q2v.q2_tiny_gemm(to_dev(g["W"].reshape(-1), dev), g["N"], g["K"], to_dev(g["A"], dev))
    n, toks = q2v.pq_verify(Y.view(S, k1, V), to_dev(v["draft"], dev), to_dev(v["drafts"], dev),
                            to_dev(v["u_acc"], dev), to_dev(v["u_fin"], dev), v["T"])
    n, toks = n.cpu().numpy(), toks.cpu().numpy()
    o = orc.pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], v["T"])
    for s in range(S):
        assert 0 <= n[s] <= k1 - 1
        assert np.array_equal(toks[s, :n[s]], v["drafts"][s, :n[s]])
        assert 0 <= toks[s, n[s]] < V and np.all(toks[s, n[s] + 1:] == -1)
        margins = [abs(float(v["u_acc"][s, i]) - o["ratio"][s, i]) for i in range(min(o["n_acc"][s] + 1, k1 - 1))
                   if np.isfinite(o["ratio"][s, i])]
        fin = min(abs(float(v["u_fin"][s]) - o["cell_lo"][s]), abs(float(v["u_fin"][s]) - o["cell_hi"][s]))
        if min(margins + [fin]) > 1e-3:
            assert n[s] == o["n_acc"][s] and np.array_equal(toks[s], o["tokens"][s]), s


# ---------------------------------------------------------------- fused vocabulary head + verify

def _fused(c, temps=None, T=None, want_probs=True, fuse=True):
    import torch
    q2v, dev, g, v = c["q2v"], c["dev"], c["g"], c["v"]
    S, k1, V = v["target"].shape
    tt = None if temps is None else torch.tensor(np.asarray(temps, np.float32), device=dev)
    probs = torch.empty((S, 2 * k1 - 1, V), dtype=torch.float32, device=dev) if want_probs else None
    ws = q2v.workspace(q2v.q2_lm_head_verify_workspace(S, k1 - 1, V, g["K"]), dev)
    tgt, n, toks = q2v.q2_lm_head_verify(to_dev(g["W"].reshape(-1), dev), V, g["K"], to_dev(g["A"], dev),
                                         to_dev(v["draft"], dev), to_dev(v["drafts"], dev), to_dev(v["u_acc"], dev),
                                         to_dev(v["u_fin"], dev), S, k1 - 1, temperatures=tt,
                                         temperature=v["T"] if T is None else T, fuse_stats=fuse, probs=probs, ws=ws)
    st = q2v.q2_get_device_status(ws)
    return (tgt.cpu().numpy(), n.cpu().numpy(), toks.cpu().numpy(),
            probs.cpu().numpy() if want_probs else None, st)


def _verify_against_oracle(c, tgt, n, toks, probs, temps=None, T=1.0):
    """The verify part against the oracle run on the GPU's own target logits."""
    v, orc = c["v"], c["orc"]
    S, k1, V = v["target"].shape
    o = orc.pq_verify(tgt, v["draft"], v["drafts"], v["u_acc"], v["u_fin"], T, temps=temps, want_probs=True)
    assert np.abs(probs.astype(np.float64) - o["probs"]).max() <= 1e-5
    greedy = np.zeros(S, bool) if temps is None else (np.asarray(temps) == 0)
    assert np.array_equal(n[greedy], o["n_acc"][greedy]) and np.array_equal(toks[greedy], o["tokens"][greedy])
    samp = np.nonzero(~greedy)[0]
    sub = {key: o[key][samp] for key in ("n_acc", "tokens", "probs", "ratio", "cell_lo", "cell_hi", "fin_src")}
    stats = compare_verify(n[samp], toks[samp], sub, v["u_acc"][samp], v["u_fin"][samp], k1 - 1)
    assert stats["exact"] + stats["mismatches_at_near_ties"] == len(samp)


@pytest.mark.parametrize("fuse", [True, False])
def test_fused_lm_head_verify(cohort, fuse):
    c = cohort
    tgt, n, toks, probs, st = _fused(c, fuse=fuse)
    assert st == 0
    S, k1, V = c["v"]["target"].shape
    check_gemm(tgt.reshape(S * k1, V), c["Yo"], c["absY"], "fused lm_head")
    _verify_against_oracle(c, tgt, n, toks, probs, T=c["v"]["T"])


def test_fused_lm_head_verify_mixed_temperatures(cohort):
    c = cohort
    S = c["v"]["target"].shape[0]
    temps = np.array([1.0, 0.0, 0.5, 2.0] * (S // 4))
    tgt, n, toks, probs, st = _fused(c, temps=temps)
    assert st == 0
    _verify_against_oracle(c, tgt, n, toks, probs, temps=temps)


@pytest.mark.parametrize("S,k,V,K", [(2, 4, 8192, 1024),    # M=10: mma.sync GEMM, unfused
                                     (4, 4, 1024, 512),     # M=20 tcgen05, small-V tier: unfused
                                     (6, 4, 20000, 512),    # M=30 tcgen05, fused, ragged last tile
                                     (1, 4, 40000, 512),    # M=5 tcgen05 (wide V), fused
                                     (2, 3, 36000, 256),    # M=8 tcgen05, fused, ragged last tile
                                     (3, 4, 20000, 256),    # M=15 tcgen05, fused
                                     (1, 4, 20000, 512)])   # M=5 narrow V: mma.sync GEMM, unfused
def test_lm_head_verify_shapes(orc, S, k, V, K):
    import torch

    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    q2v.load()
    dev = torch.device("cuda:0")
    st = synth.Streams(800 + S * 31 + V)
    W = synth.q2b32_weights(st, V, K)
    A = synth.activations_bf16(st, S * (k + 1), K)
    Yo, absY = orc.gemm(W, V, K, A)
    v = synth.verify_inputs(st, S, k, V, 0.0, 1.0, 1.0, target=Yo.astype(np.float32).reshape(S, k + 1, V))
    probs = torch.empty((S, 2 * k + 1, V), dtype=torch.float32, device=dev)
    tgt, n, toks = q2v.q2_lm_head_verify(to_dev(W.reshape(-1), dev), V, K, to_dev(A, dev), to_dev(v["draft"], dev),
                                         to_dev(v["drafts"], dev), to_dev(v["u_acc"], dev), to_dev(v["u_fin"], dev),
                                         S, k, temperature=1.0, fuse_stats=True, probs=probs)
    tgt = tgt.cpu().numpy()
    check_gemm(tgt.reshape(S * (k + 1), V), Yo, absY, f"lm_head S={S} V={V}")
    c = dict(v=v, orc=orc)
    _verify_against_oracle(c, tgt, n.cpu().numpy(), toks.cpu().numpy(), probs.cpu().numpy(), T=1.0)
