"""pq_verify on the GPU against the fp64 oracle: accepted counts and tokens identical except
at counted near-ties, probabilities within 1e-5, and the chi-square law of the emitted
tokens at V=16 over 1e6 sessions."""
import numpy as np
import pytest

from _util import PROB_ATOL, compare_verify, to_dev
from speculative_decode_verifier_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(orc):
    import torch

    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    q2v.load()
    return torch.device("cuda:0"), q2v, orc


def _gpu(env, v, want_probs=False, ws=None):
    import torch
    dev, q2v, _ = env
    S, k1, V = v["target"].shape
    k = k1 - 1
    t = {n: to_dev(v[n], dev) for n in ("target", "draft", "drafts", "u_acc", "u_fin")}
    probs = torch.empty((S, 2 * k + 1, V), dtype=torch.float32, device=dev) if want_probs else None
    n_acc, toks = q2v.pq_verify(t["target"], t["draft"] if k else None, t["drafts"] if k else None,
                                t["u_acc"] if k else None, t["u_fin"], v["T"], probs=probs, ws=ws)
    return n_acc.cpu().numpy(), toks.cpu().numpy(), (probs.cpu().numpy() if want_probs else None)


def _check(env, v, want_probs=True, report=None):
    n, toks, probs = _gpu(env, v, want_probs)
    o = env[2].pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], v["T"], want_probs=True)
    k = v["target"].shape[1] - 1
    if want_probs:
        err = np.abs(probs.astype(np.float64) - o["probs"])
        assert err.max() <= PROB_ATOL, err.max()
    stats = compare_verify(n, toks, o, v["u_acc"], v["u_fin"], k)
    if report is not None:
        report.append(stats)
    # structural checks that hold for any correct result
    assert np.all((n >= 0) & (n <= k))
    for s in range(n.shape[0]):
        assert np.array_equal(toks[s, :n[s]], v["drafts"][s, :n[s]])
        assert 0 <= toks[s, n[s]] < v["target"].shape[2]
        assert np.all(toks[s, n[s] + 1:] == -1)
    return stats


def test_tiny_smoke_config(env):
    _check(env, synth.config_verify(0))


def test_batched_config_full_size(env):
    # S=3, k=4, V=129280: the split (multi-CTA) tier
    stats = _check(env, synth.config_verify(3))
    assert stats["exact"] + stats["mismatches_at_near_ties"] == 3


@pytest.mark.parametrize("S,k,V,T", [
    (64, 4, 1024, 1.0),      # small-V tier (a CTA per session), many sessions
    (5, 4, 4096, 0.7),       # largest small-V tier V: 16 tokens per thread in the draw
    (3, 16, 512, 1.0),       # largest V of one warp per session, the largest k (33 rows in one warp)
    (6, 4, 513, 1.0),        # smallest V of a CTA per session, V % 4 != 0 (scalar loads)
    (11, 3, 17, 0.8),        # one warp per session, scalar loads, 1 token per lane in the draw
    (2, 16, 4000, 1.2),      # a CTA per session with 33 rows over 8 warps
    (5, 4, 4097, 1.0),       # smallest split-tier V, V % 4 != 0 (scalar loads)
    (7, 3, 10000, 1.5),      # ragged last chunk
    (40, 4, 32768, 1.0),     # many sessions: few chunks each
    (320, 2, 20000, 1.0),    # one chunk per session: segments of 2,512 tokens, 10 per thread in the draw
    (2, 16, 8192, 1.0),      # the largest k
    (3, 0, 5000, 1.0),       # k = 0: plain sampling from p_0
    (9, 0, 300, 0.9),        # k = 0 in the small-V tier
    (4, 2, 1, 1.0),          # V = 1
    (4, 4, 129280, 50.0),    # near-uniform p and q: CDF cells ~7.7e-6 wide, residuals of nearly equal probabilities
])
def test_shapes(env, S, k, V, T):
    st = synth.Streams(5000 + S + 31 * k + V)
    v = synth.verify_inputs(st, S, k, V, t_std=2.0, noise_std=0.7, T=T)
    _check(env, v)


def test_p_equals_q_accepts_everything(env):
    v = synth.config_verify(3)
    v["draft"] = np.ascontiguousarray(v["target"][:, :4])
    n, toks, _ = _gpu(env, v)
    assert np.all(n == 4)
    _check(env, v, want_probs=False)


def test_masked_vocabulary(env):
    """-inf logits (a masked vocabulary) have probability 0 and are never emitted."""
    st = synth.Streams(91)
    for V in (2048, 20000):
        v = synth.verify_inputs(st, 4, 3, V, t_std=2.0, noise_std=0.5, T=1.0)
        mask = st["extra0"].random(V) < 0.3
        mask[:4] = True
        v["target"][:, :, mask] = -np.inf
        v["draft"][:, :, mask] = -np.inf
        v["drafts"] = synth.gumbel_max_drafts(v["draft"], 1.0, st["extra1"])
        _check(env, v)
        n, toks, _ = _gpu(env, v)
        for s in range(4):
            assert not mask[toks[s, n[s]]]


def test_bad_token_sets_status(env):
    dev, q2v, _ = env
    for V, bad in ((1024, None), (8192, None), (1024, -1), (8192, -1)):
        v = synth.config_verify(0, V=V, S=3)
        v["drafts"] = v["drafts"].copy()
        v["drafts"][1, 2] = V if bad is None else bad
        ws = q2v.workspace(q2v.pq_verify_workspace(3, 4, V), dev)
        n, toks, _ = _gpu(env, v, ws=ws)
        assert q2v.q2_get_device_status(ws) == 7  # Q2_ERR_BAD_TOKEN
        assert n[1] == -1 and np.all(toks[1] == -1)
        assert n[0] >= 0 and n[2] >= 0  # the other sessions are verified as usual
        assert q2v.q2_get_device_status(ws) == 0


def test_repeated_calls_reuse_workspace(env):
    dev, q2v, _ = env
    v = synth.config_verify(3)
    ws = q2v.workspace(q2v.pq_verify_workspace(3, 4, 129280), dev)
    a = _gpu(env, v, ws=ws)
    b = _gpu(env, v, ws=ws)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_chi_square_emitted_law_on_gpu(env):
    """1e6 sessions at V=16: the token at position i (given n_acc >= i) is distributed as p_i;
    also every session matches the oracle outside near-ties."""
    import scipy.stats
    S, k, V, T = 1_000_000, 4, 16, 1.0
    st = synth.Streams(synth.SEED0 + 177)
    tl1 = st["t_logits"].normal(0, 1.0, size=(k + 1, V)).astype(np.float32)
    dl1 = (tl1[:k] + st["noise"].normal(0, 1.0, size=(k, V))).astype(np.float32)
    v = dict(target=np.ascontiguousarray(np.broadcast_to(tl1, (S, k + 1, V))),
             draft=np.ascontiguousarray(np.broadcast_to(dl1, (S, k, V))), T=T)
    v["drafts"] = synth.gumbel_max_drafts(v["draft"], T, st["draft_uniforms"])
    v["u_acc"] = synth.uniforms_f32(st["u_acc"], (S, k))
    v["u_fin"] = synth.uniforms_f32(st["u_fin"], (S,))
    n, toks, _ = _gpu(env, v)
    import scipy.special
    p = scipy.special.softmax(tl1.astype(np.float64) / T, axis=-1)
    for i in range(k + 1):
        sel = n >= i
        counts = np.bincount(toks[sel, i], minlength=V).astype(np.float64)
        exp = counts.sum() * p[i]
        stat = ((counts - exp) ** 2 / exp).sum()
        assert scipy.stats.chi2.sf(stat, df=V - 1) > 1e-3, i
    o = env[2].pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], T)
    o["probs"] = None
    diff = np.nonzero((n != o["n_acc"]) | np.any(toks != o["tokens"], axis=1))[0]
    sub = lambda a: a[diff]  # noqa: E731
    if diff.size:
        stats = compare_verify(n[diff], toks[diff], {kk: (sub(vv) if isinstance(vv, np.ndarray) else vv)
                                                     for kk, vv in o.items()},
                               v["u_acc"][diff], v["u_fin"][diff], k)
        assert stats["mismatches_at_near_ties"] == diff.size
    assert diff.size <= 200


# ---------------------------------------------------------------- per-session temperature, greedy

def _gpu_ex(env, v, temps, want_probs=False):
    import torch
    dev, q2v, _ = env
    S, k1, V = v["target"].shape
    k = k1 - 1
    t = {n: to_dev(v[n], dev) for n in ("target", "draft", "drafts", "u_acc", "u_fin")}
    tt = torch.tensor(np.asarray(temps, np.float32), device=dev)
    probs = torch.empty((S, 2 * k + 1, V), dtype=torch.float32, device=dev) if want_probs else None
    ws = q2v.workspace(q2v.pq_verify_workspace(S, k, V), dev)
    n_acc, toks = q2v.pq_verify_ex(t["target"], t["draft"] if k else None, t["drafts"] if k else None,
                                   t["u_acc"] if k else None, t["u_fin"], tt, probs=probs, ws=ws)
    st = q2v.q2_get_device_status(ws)
    return n_acc.cpu().numpy(), toks.cpu().numpy(), (probs.cpu().numpy() if want_probs else None), st


def _greedy_inputs(seed, S, k, V):
    """Seeded logits whose drafts agree with the target argmax for a random prefix."""
    st = synth.Streams(seed)
    v = synth.verify_inputs(st, S, k, V, 3.0, 1.0, 1.0)
    am = np.argmax(v["target"], axis=2)
    rng = np.random.default_rng(seed)
    for s in range(S):
        agree = rng.integers(0, k + 1)
        v["drafts"][s, :agree] = am[s, :agree]
    return v


@pytest.mark.parametrize("S,k,V", [(8, 4, 1024), (3, 4, 129280), (5, 3, 8192), (4, 0, 5000)])
def test_greedy_matches_oracle_exactly(env, S, k, V):
    v = _greedy_inputs(400 + V, S, k, V)
    n, toks, probs, st = _gpu_ex(env, v, np.zeros(S), want_probs=True)
    o = env[2].pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], 1.0, temps=np.zeros(S),
                         want_probs=True)
    assert st == 0
    assert np.array_equal(n, o["n_acc"]) and np.array_equal(toks, o["tokens"])
    assert np.array_equal(probs.astype(np.float64), o["probs"])  # one-hot rows
    assert n.max() > 0 or k == 0


@pytest.mark.parametrize("V", [1024, 8192, 129280])
def test_mixed_temperatures_match_oracle(env, V):
    S, k = 6, 4
    v = synth.verify_inputs(synth.Streams(500 + V), S, k, V, 3.0, 1.0, 1.0)
    temps = np.array([0.5, 1.0, 0.0, 2.0, 0.0, 1.3])
    n, toks, probs, st = _gpu_ex(env, v, temps, want_probs=True)
    o = env[2].pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], 1.0, temps=temps,
                         want_probs=True)
    assert st == 0
    assert np.abs(probs.astype(np.float64) - o["probs"]).max() <= PROB_ATOL
    greedy = temps == 0.0
    assert np.array_equal(n[greedy], o["n_acc"][greedy]) and np.array_equal(toks[greedy], o["tokens"][greedy])
    samp = np.nonzero(~greedy)[0]
    sub = {key: (o[key][samp] if o[key] is not None else None) for key in o if key not in ("bad_token", "bad_temperature")}
    stats = compare_verify(n[samp], toks[samp], sub, v["u_acc"][samp], v["u_fin"][samp], k)
    assert stats["exact"] + stats["mismatches_at_near_ties"] == len(samp)


@pytest.mark.parametrize("V", [1024, 129280])
def test_bad_temperature_marks_only_its_session(env, V):
    S, k = 4, 3
    v = synth.verify_inputs(synth.Streams(600 + V), S, k, V, 3.0, 1.0, 1.0)
    temps = np.array([1.0, -0.5, np.nan, 0.0])
    n, toks, _, st = _gpu_ex(env, v, temps)
    assert st == 9  # Q2_ERR_BAD_TEMPERATURE
    assert list(n[1:3]) == [-1, -1] and np.all(toks[1:3] == -1)
    o = env[2].pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], 1.0, temps=temps,
                         want_probs=True)
    assert n[3] == o["n_acc"][3] and np.array_equal(toks[3], o["tokens"][3])
    sub = {key: (o[key][[0]] if o[key] is not None else None) for key in o if key not in ("bad_token", "bad_temperature")}
    stats = compare_verify(n[[0]], toks[[0]], sub, v["u_acc"][[0]], v["u_fin"][[0]], k)
    assert stats["exact"] + stats["mismatches_at_near_ties"] == 1


@pytest.mark.parametrize("V", [1024, 129280])
def test_equal_temperatures_equal_the_scalar_call(env, V):
    S, k = 3, 4
    v = synth.verify_inputs(synth.Streams(700 + V), S, k, V, 3.0, 1.0, 1.0)
    v["T"] = 0.8
    n0, t0, p0 = _gpu(env, v, want_probs=True)
    n1, t1, p1, st = _gpu_ex(env, v, np.full(S, 0.8), want_probs=True)
    assert st == 0 and np.array_equal(n0, n1) and np.array_equal(t0, t1) and np.array_equal(p0, p1)
