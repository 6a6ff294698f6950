"""Pins of the fp64 oracle against things other than itself: format fixtures derived by
hand, library routines (numpy/scipy/torch), closed forms, special cases and brute-force
enumeration.  CPU only."""
import os

import numpy as np
import pytest
import scipy.special

from speculative_decode_verifier_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- number formats

def test_half_decode_matches_numpy_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_matches_torch_all_patterns(orc):
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.int32).astype(np.int16)
    ref = torch.from_numpy(bits).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_to_f64(int(b) & 0xFFFF) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _read_golden_rows():
    vals = {}
    with open(os.path.join(GOLDEN, "q2b32_rows.txt")) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = rest.split()
    W = np.array([int(x, 16) for x in vals["bytes"]], np.uint8)
    codes = np.array([int(x) for x in vals["codes"]])
    d = np.array([float(x) for x in vals["scale_d"]])
    m = np.array([float(x) for x in vals["offset_m"]])
    return W, codes, d, m


def test_q2b32_golden_block_layout(orc):
    W, codes, d, m = _read_golden_rows()
    K = codes.size
    got = orc.dequant(W, 1, K)[0]
    blk = np.arange(K) // 32
    expect = d[blk] * codes + m[blk]
    assert np.array_equal(got, expect)


def test_q2b32_every_code_at_every_position(orc):
    # brute force over all 4 codes in each of the 32 slots of a single-block row
    d_bits = synth.fp16_bits(np.array([0.25]))[0]
    m_bits = synth.fp16_bits(np.array([0.125]))[0]
    for j in range(32):
        for c in range(4):
            codes = np.zeros((1, 32), np.uint8)
            codes[0, j] = c
            W = synth.pack_q2b32(codes, np.array([[d_bits]]), np.array([[m_bits]]))
            w = orc.dequant(W, 1, 32)[0]
            expect = np.full(32, 0.125)
            expect[j] = 0.25 * c + 0.125
            assert np.array_equal(w, expect), (j, c)


def test_pack_q2b32_matches_golden_bytes():
    W, codes, d, m = _read_golden_rows()
    d_bits = synth.fp16_bits(d).reshape(1, 2)
    m_bits = synth.fp16_bits(m).reshape(1, 2)
    packed = synth.pack_q2b32(codes.reshape(1, 64).astype(np.uint8), d_bits, m_bits)
    assert np.array_equal(packed.reshape(-1), W)


# ----------------------------------------------------------------- GEMM

def _rand_gemm(seed, M, N, K):
    st = synth.Streams(seed)
    W = synth.q2b32_weights(st, N, K)
    A = synth.activations_bf16(st, M, K)
    return W, A


@pytest.mark.parametrize("M,N,K", [(1, 3, 32), (3, 7, 64), (5, 16, 256), (4, 33, 96)])
def test_gemm_matches_numpy_matmul(orc, M, N, K):
    W, A = _rand_gemm(11 + M * N, M, N, K)
    Wd = orc.dequant(W, N, K)
    Af = synth.bf16_bits_to_f32(A).astype(np.float64)
    Y, absY = orc.gemm(W, N, K, A)
    ref = Af @ Wd.T
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(absY, np.abs(Af[:, None, :] * Wd[None, :, :]).sum(-1), rtol=1e-12)


def test_gemm_special_case_zero_scale(orc):
    # d = 0  =>  Y[m,n] = sum over blocks of m_{n,b} * (sum of A over the block)
    st = synth.Streams(5)
    M, N, K = 3, 5, 128
    codes = st["codes"].integers(0, 4, size=(N, K), dtype=np.uint8)
    d_bits = np.zeros((N, K // 32), np.uint16)
    mvals = st["m"].normal(0, 0.5, size=(N, K // 32))
    m_bits = synth.fp16_bits(mvals)
    W = synth.pack_q2b32(codes, d_bits, m_bits)
    A = synth.activations_bf16(st, M, K)
    Af = synth.bf16_bits_to_f32(A).astype(np.float64)
    mv = m_bits.view(np.float16).astype(np.float64)
    blocksum = Af.reshape(M, K // 32, 32).sum(-1)
    Y, _ = orc.gemm(W, N, K, A)
    np.testing.assert_allclose(Y, blocksum @ mv.T, rtol=1e-12, atol=1e-14)


def test_gemm_special_case_all_threes(orc):
    # all codes 3, d = 1, m = 0  =>  Y = 3 * sum_k A
    st = synth.Streams(6)
    M, N, K = 4, 6, 256
    codes = np.full((N, K), 3, np.uint8)
    W = synth.pack_q2b32(codes, synth.fp16_bits(np.ones((N, K // 32))),
                         synth.fp16_bits(np.zeros((N, K // 32))))
    A = synth.activations_bf16(st, M, K)
    Af = synth.bf16_bits_to_f32(A).astype(np.float64)
    Y, _ = orc.gemm(W, N, K, A)
    assert np.array_equal(Y, np.repeat((3 * Af.sum(1))[:, None], N, 1))


def test_gemm_special_case_one_hot(orc):
    # a one-hot activation row picks out one dequantised column exactly
    W, _ = _rand_gemm(7, 1, 9, 96)
    Wd = orc.dequant(W, 9, 96)
    for k0 in (0, 31, 32, 95):
        a = np.zeros((1, 96))
        a[0, k0] = 1.0
        Y, _ = orc.gemm(W, 9, 96, synth.bf16_bits(a))
        assert np.array_equal(Y[0], Wd[:, k0])


# ----------------------------------------------------------------- softmax / sampling

def test_softmax_matches_scipy(orc):
    rng = np.random.default_rng(3)
    for T in (0.5, 1.0, 1.7):
        x = rng.normal(0, 4, size=1000).astype(np.float32)
        ref = scipy.special.softmax(x.astype(np.float64) / T)
        np.testing.assert_allclose(orc.softmax(x, T), ref, rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(orc.softmax(np.zeros(16, np.float32)), np.full(16, 1 / 16), rtol=0)


def test_inverse_cdf_matches_searchsorted(orc):
    rng = np.random.default_rng(4)
    for _ in range(200):
        V = int(rng.integers(1, 40))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[0] = 1.0
        u = float(rng.random())
        y, lo, hi = orc.inverse_cdf(w, u)
        c = np.cumsum(w)
        assert y == int(np.searchsorted(c, u * c[-1], side="right"))
        assert w[y] > 0 and lo <= u < hi or np.isclose(lo, u) or np.isclose(hi, u)
    assert orc.inverse_cdf(np.array([1.0, 1.0, 1.0, 1.0]), 0.3)[0] == 1
    assert orc.inverse_cdf(np.array([0.0, 0.0, 2.0, 1.0]), 0.0)[0] == 2
    assert orc.inverse_cdf(np.zeros(3), 0.5)[0] == -1


# ----------------------------------------------------------------- p/q verify: brute force

def _softmax_rows(x, T):
    return scipy.special.softmax(np.asarray(x, np.float64) / T, axis=-1)


def _theory_law(p, q):
    """Exact law of (n_acc, emitted tokens) of speculative sampling with drafts x_i ~ q_i,
    acceptance min(1, p/q), residual max(0, p-q) (p if that is zero), bonus from p_k.
    p: [k+1, V], q: [k, V].  Returns {(n_acc, tokens tuple): probability}."""
    k, V = q.shape
    law = {}

    def rec(i, prefix, prob):
        if i == k:
            for y in range(V):
                key = (k, tuple(prefix) + (y,))
                law[key] = law.get(key, 0.0) + prob * p[k, y]
            return
        acc = np.minimum(1.0, np.divide(p[i], q[i], out=np.full(V, np.inf), where=q[i] > 0))
        rej_mass = float(np.sum(q[i] * (1.0 - acc)))
        res = np.maximum(p[i] - q[i], 0.0)
        res = res / res.sum() if res.sum() > 0 else p[i]
        for y in range(V):
            if rej_mass > 0 and res[y] > 0:
                key = (i, tuple(prefix) + (y,))
                law[key] = law.get(key, 0.0) + prob * rej_mass * res[y]
        for x in range(V):
            if q[i, x] > 0 and acc[x] > 0:
                rec(i + 1, prefix + [x], prob * q[i, x] * acc[x])

    rec(0, [], 1.0)
    return law


def _oracle_law(orc, tl, dl, T):
    """Law of the oracle's output when drafts ~ q and the uniforms are uniform: enumerate
    every draft tuple and every cell of the uniforms on which the output is constant."""
    k1, V = tl.shape
    k = k1 - 1
    p = _softmax_rows(tl, T)
    q = _softmax_rows(dl, T) if k else np.zeros((0, V))
    # breakpoints of u_fin: normalised CDFs of every distribution a final draw may use
    bps = {0.0, 1.0}
    dists = [p[k]] + [np.maximum(p[j] - q[j], 0) for j in range(k)] + [p[j] for j in range(k)]
    for w in dists:
        if w.sum() > 0:
            bps.update(np.cumsum(w) / w.sum())
    bps = np.array(sorted(b for b in bps if 0.0 <= b <= 1.0))
    mids = (bps[:-1] + bps[1:]) / 2
    lens = np.diff(bps)
    keep = lens > 1e-15
    mids, lens = mids[keep], lens[keep]
    law = {}
    import itertools
    for xs in itertools.product(range(V), repeat=k):
        wx = np.prod([q[i, xs[i]] for i in range(k)]) if k else 1.0
        if wx == 0:
            continue
        # u_acc cells: [0, r) accepts, [r, 1) rejects
        r = [p[i, xs[i]] / q[i, xs[i]] for i in range(k)]
        acc_cells = []
        for i in range(k):
            cells = []
            if r[i] > 0:
                cells.append((min(r[i], 1.0) / 2, min(r[i], 1.0)))
            if r[i] < 1:
                cells.append(((r[i] + 1) / 2, 1 - r[i]))
            acc_cells.append(cells)
        for combo in itertools.product(*acc_cells) if k else [()]:
            wa = np.prod([c[1] for c in combo]) if k else 1.0
            S = mids.size
            tgt = np.broadcast_to(tl, (S, k + 1, V))
            drf = np.broadcast_to(dl, (S, k, V)) if k else np.zeros((S, 0, V), np.float32)
            out = orc.pq_verify(tgt, drf, np.tile(np.array(xs, np.int32), (S, 1)),
                                np.tile(np.array([c[0] for c in combo], np.float32), (S, 1)),
                                mids.astype(np.float32), T, threads=1)
            for s in range(S):
                n = int(out["n_acc"][s])
                key = (n, tuple(int(t) for t in out["tokens"][s, :n + 1]))
                law[key] = law.get(key, 0.0) + wx * wa * lens[s]
    return law


@pytest.mark.parametrize("V,k,seed", [(2, 1, 0), (3, 1, 1), (3, 2, 2), (4, 2, 3), (4, 0, 4), (2, 2, 5)])
def test_pq_verify_brute_force_law(orc, V, k, seed):
    rng = np.random.default_rng(100 + seed)
    T = 1.0 if seed % 2 == 0 else 0.8
    # quantise logits to multiples of 1/8 so that fp32 storage is exact and the u cells
    # do not sit on fp32 rounding boundaries
    tl = (np.round(rng.normal(0, 1.5, size=(k + 1, V)) * 8) / 8).astype(np.float32)
    dl = (tl[:k] + np.round(rng.normal(0, 1.0, size=(k, V)) * 8) / 8).astype(np.float32)
    theory = _theory_law(_softmax_rows(tl, T), _softmax_rows(dl, T) if k else np.zeros((0, V)))
    got = _oracle_law(orc, tl, dl, T)
    keys = set(theory) | set(got)
    for key in keys:
        assert abs(theory.get(key, 0.0) - got.get(key, 0.0)) < 1e-6, (key, theory.get(key), got.get(key))
    # the invariant the pages fix: the first emitted token is distributed as p_0
    p0 = _softmax_rows(tl[0], T)
    marg = np.zeros(V)
    for (n, toks), pr in got.items():
        marg[toks[0]] += pr
    np.testing.assert_allclose(marg, p0, atol=1e-6)


# ----------------------------------------------------------------- p/q verify: special cases

def test_pq_verify_p_equals_q_accepts_all(orc):
    v = synth.config_verify(0)
    tl = v["target"]
    dl = tl[:, :4].copy()
    out = orc.pq_verify(tl, dl, v["drafts"], v["u_acc"], v["u_fin"], 1.0)
    assert out["n_acc"][0] == 4
    assert out["fin_src"][0] == 1
    p4 = _softmax_rows(tl[0, 4], 1.0)
    y = int(np.searchsorted(np.cumsum(p4), float(v["u_fin"][0]) * p4.sum(), side="right"))
    assert out["tokens"][0, 4] == y


def test_pq_verify_onehot_q_zero_p_always_rejects(orc):
    V, k = 8, 2
    rng = np.random.default_rng(9)
    tl = rng.normal(0, 1, size=(1, k + 1, V)).astype(np.float32)
    tl[0, 0, 3] = -1e4            # p_0(3) underflows to exactly 0
    dl = np.full((1, k, V), -1e4, np.float32)
    dl[0, :, 3] = 0.0             # q_i one-hot on token 3
    for u in (0.0, 0.3, 0.999):
        out = orc.pq_verify(tl, dl, np.array([[3, 3]]), np.array([[0.0, 0.0]]),
                            np.array([u], np.float32), 1.0)
        assert out["n_acc"][0] == 0
        p0 = _softmax_rows(tl[0, 0], 1.0)
        y = int(np.searchsorted(np.cumsum(p0), np.float32(u) * p0.sum(), side="right"))
        assert out["tokens"][0, 0] == y and y != 3
        assert list(out["tokens"][0, 1:]) == [-1, -1]


def test_pq_verify_k0_is_plain_sampling(orc):
    rng = np.random.default_rng(12)
    V = 50
    tl = rng.normal(0, 2, size=(6, 1, V)).astype(np.float32)
    u = synth.uniforms_f32(rng, (6,))
    out = orc.pq_verify(tl, np.zeros((6, 0, V), np.float32), np.zeros((6, 0), np.int32),
                        np.zeros((6, 0), np.float32), u, 1.3)
    for s in range(6):
        p = _softmax_rows(tl[s, 0], 1.3)
        assert out["tokens"][s, 0] == np.searchsorted(np.cumsum(p), float(u[s]) * p.sum(), side="right")
    assert np.all(out["n_acc"] == 0)


def test_pq_verify_rejects_bad_token(orc):
    v = synth.config_verify(0)
    drafts = v["drafts"].copy()
    drafts[0, 2] = 1024
    out = orc.pq_verify(v["target"], v["draft"], drafts, v["u_acc"], v["u_fin"], 1.0)
    assert out["bad_token"] and out["n_acc"][0] == -1


# ----------------------------------------------------------------- p/q verify: statistics

def _chi2_sf(counts, probs):
    n = counts.sum()
    exp = n * probs
    stat = float(((counts - exp) ** 2 / exp).sum())
    return scipy.stats.chi2.sf(stat, df=len(probs) - 1)


def test_pq_verify_chi_square_emitted_law(orc):
    import scipy.stats  # noqa: F401
    S, k, V, T = 1_000_000, 4, 16, 1.0
    st = synth.Streams(synth.SEED0 + 77)
    tl1 = st["t_logits"].normal(0, 1.0, size=(k + 1, V)).astype(np.float32)
    dl1 = (tl1[:k] + st["noise"].normal(0, 1.0, size=(k, V))).astype(np.float32)
    tl = np.broadcast_to(tl1, (S, k + 1, V))
    dl = np.broadcast_to(dl1, (S, k, V))
    drafts = synth.gumbel_max_drafts(dl, T, st["draft_uniforms"])
    u_acc = synth.uniforms_f32(st["u_acc"], (S, k))
    u_fin = synth.uniforms_f32(st["u_fin"], (S,))
    out = orc.pq_verify(tl, dl, drafts, u_acc, u_fin, T)
    p = _softmax_rows(tl1, T)
    q = _softmax_rows(dl1, T)
    n_acc, toks = out["n_acc"], out["tokens"]
    for i in range(k + 1):
        sel = n_acc >= i
        counts = np.bincount(toks[sel, i], minlength=V).astype(np.float64)
        assert _chi2_sf(counts, p[i]) > 1e-3, i
    # closed forms: acceptance rate alpha_i = sum min(p_i, q_i); E[n_acc] = sum_i prod_{j<i} alpha_j
    alpha = np.minimum(p[:k], q).sum(-1)
    e_nacc = sum(np.prod(alpha[:i]) for i in range(1, k + 1))
    sd = n_acc.std() / np.sqrt(S)
    assert abs(n_acc.mean() - e_nacc) < 5 * sd
    rate0 = (n_acc >= 1).mean()
    assert abs(rate0 - alpha[0]) < 5 * np.sqrt(alpha[0] * (1 - alpha[0]) / S)
    pk = np.prod(alpha)
    assert abs((n_acc == k).mean() - pk) < 5 * np.sqrt(pk * (1 - pk) / S)


def test_chi_square_detects_a_planted_mistake(orc):
    """The statistical pin has power: a verifier that skips the residual (resamples from
    p instead of max(0, p - q)) is rejected by the same chi-square test."""
    import scipy.stats  # noqa: F401
    S, k, V, T = 200_000, 1, 16, 1.0
    rng = np.random.default_rng(31)
    tl1 = rng.normal(0, 1.0, size=(k + 1, V))
    dl1 = tl1[:k] + rng.normal(0, 1.0, size=(k, V))
    p = _softmax_rows(tl1, T)
    q = _softmax_rows(dl1, T)
    x = synth.gumbel_max_drafts(np.broadcast_to(dl1, (S, k, V)), T, rng)[:, 0]
    u = rng.random(S)
    acc = u < p[0, x] / q[0, x]
    uf = rng.random(S)
    wrong = np.where(acc, x, np.searchsorted(np.cumsum(p[0]), uf, side="right").clip(0, V - 1))
    counts = np.bincount(wrong, minlength=V).astype(np.float64)
    assert _chi2_sf(counts, p[0]) < 1e-3


# ----------------------------------------------------------------- MoE

def _silu(z):
    # z * sigmoid(z) through scipy's logistic function, not the oracle's own expression
    return z * scipy.special.expit(z)


def test_silu_reference_identities():
    # silu(z) - silu(-z) = z (sigmoid(z) + sigmoid(-z) = 1), silu(0) = 0, silu(z) -> z for large z
    z = np.linspace(-30.0, 30.0, 601)
    np.testing.assert_allclose(_silu(z) - _silu(-z), z, rtol=0, atol=1e-12)
    assert _silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(_silu(np.array([40.0])), [40.0], rtol=1e-15)


def test_moe_single_expert_reduces_to_three_gemms(orc):
    st = synth.Streams(21)
    H, F = 64, 96
    Wg = synth.q2b32_weights(st, F, H)
    Wu = synth.q2b32_weights(st, F, H)
    Wd = synth.q2b32_weights(st, H, F)
    X = synth.activations_bf16(st, 1, H)
    out = orc.moe(Wg, Wu, Wd, 1, H, F, 1, X, np.zeros((1, 1), np.float32))
    x = synth.bf16_bits_to_f32(X).astype(np.float64)[0]
    g = orc.dequant(Wg, F, H) @ x
    u = orc.dequant(Wu, F, H) @ x
    y = orc.dequant(Wd, H, F) @ (_silu(g) * u)
    np.testing.assert_allclose(out["Y"][0], y, rtol=1e-11, atol=1e-13)
    assert out["ids"][0, 0] == 0 and out["weights"][0, 0] == 1.0


@pytest.mark.parametrize("renorm", [False, True])
def test_moe_routing_and_combine_brute_force(orc, renorm):
    st = synth.Streams(22)
    E, H, F, M, topk = 4, 32, 64, 3, 2
    Wg = synth.q2b32_weights(st, F, H, batch=E)
    Wu = synth.q2b32_weights(st, F, H, batch=E)
    Wd = synth.q2b32_weights(st, H, F, batch=E)
    X = synth.activations_bf16(st, M, H)
    router = st["router"].normal(0, 1, size=(M, E)).astype(np.float32)
    router[2, 1] = router[2, 3]          # a tie: the lower index must win
    out = orc.moe(Wg, Wu, Wd, E, H, F, topk, X, router, renorm=renorm)
    x = synth.bf16_bits_to_f32(X).astype(np.float64)
    gq = orc.dequant(Wg, E * F, H).reshape(E, F, H)
    uq = orc.dequant(Wu, E * F, H).reshape(E, F, H)
    dq = orc.dequant(Wd, E * H, F).reshape(E, H, F)
    for r in range(M):
        prob = scipy.special.softmax(router[r].astype(np.float64))
        ids = np.argsort(-prob, kind="stable")[:topk]
        assert list(out["ids"][r]) == list(ids)
        w = prob[ids] / (prob[ids].sum() if renorm else 1.0)
        np.testing.assert_allclose(out["weights"][r], w, rtol=1e-14)
        y = sum(w[t] * (dq[e] @ (_silu(gq[e] @ x[r]) * (uq[e] @ x[r]))) for t, e in enumerate(ids))
        np.testing.assert_allclose(out["Y"][r], y, rtol=1e-11, atol=1e-13)
        assert np.all(out["tol"][r] > 0)


def _silu_derivative():
    """d silu / dz, differentiated symbolically by sympy from z / (1 + exp(-z)) (not the
    oracle's closed form), as a numpy function."""
    sympy = pytest.importorskip("sympy")
    z = sympy.Symbol("z", real=True)
    return sympy.lambdify(z, sympy.diff(z / (1 + sympy.exp(-z)), z), "numpy")


def _moe_tol_numpy(gq, uq, dq, ids, w, x, rel=2e-3):
    """The MoE parity bound from its definition, with numpy matrix products: per output n,
    sum over the row's slots of g * (rel * sum_f |h_f wd_nf| + sum_f |wd_nf| dh_f), where
    dh_f = |d silu(gate_f)/d gate * up_f| * tol_gate_f + |silu(gate_f)| * tol_up_f and tol_gate,
    tol_up are the GEMM bounds rel * sum_k |x_k w_fk| of the gate and up projections."""
    dsilu = _silu_derivative()
    tol = np.zeros(dq.shape[1])
    for t, e in enumerate(ids):
        gate, up = gq[e] @ x, uq[e] @ x
        tg, tu = rel * (np.abs(gq[e]) @ np.abs(x)), rel * (np.abs(uq[e]) @ np.abs(x))
        h = _silu(gate) * up
        dh = np.abs(dsilu(gate) * up) * tg + np.abs(_silu(gate)) * tu
        tol += w[t] * (rel * (np.abs(dq[e]) @ np.abs(h)) + np.abs(dq[e]) @ dh)
    return tol


def test_silu_derivative_reference_matches_finite_differences():
    dsilu = _silu_derivative()
    z = np.linspace(-12.0, 12.0, 97)
    eps = 1e-6
    fd = (_silu(z + eps) - _silu(z - eps)) / (2 * eps)
    np.testing.assert_allclose(dsilu(z), fd, rtol=0, atol=1e-8)


@pytest.mark.parametrize("renorm", [False, True])
def test_moe_tolerance_matches_its_definition(orc, renorm):
    """The oracle's MoE bound `tol` equals the bound recomputed from its definition (the GEMM
    rule 2e-3 * sum |a w| carried through silu(gate) * up to first order, then through the down
    projection and the gate weights) on the brute-force routing case; a dropped gate weight,
    a wrong derivative or a 10x relative factor would each change it far beyond 1e-12."""
    st = synth.Streams(22)
    E, H, F, M, topk = 4, 32, 64, 3, 2
    Wg = synth.q2b32_weights(st, F, H, batch=E)
    Wu = synth.q2b32_weights(st, F, H, batch=E)
    Wd = synth.q2b32_weights(st, H, F, batch=E)
    X = synth.activations_bf16(st, M, H)
    router = st["router"].normal(0, 1, size=(M, E)).astype(np.float32)
    out = orc.moe(Wg, Wu, Wd, E, H, F, topk, X, router, renorm=renorm)
    x = synth.bf16_bits_to_f32(X).astype(np.float64)
    gq = orc.dequant(Wg, E * F, H).reshape(E, F, H)
    uq = orc.dequant(Wu, E * F, H).reshape(E, F, H)
    dq = orc.dequant(Wd, E * H, F).reshape(E, H, F)
    for r in range(M):
        prob = scipy.special.softmax(router[r].astype(np.float64))
        ids = np.argsort(-prob, kind="stable")[:topk]
        w = prob[ids] / (prob[ids].sum() if renorm else 1.0)
        want = _moe_tol_numpy(gq, uq, dq, ids, w, x[r])
        np.testing.assert_allclose(out["tol"][r], want, rtol=1e-12, atol=0)


def _q2b32_constant_rows(n_rows, K, code, d_bits, m_bits=0):
    """Q2B32 bytes of n_rows x K weights, every code equal to `code`, scale and offset given as
    fp16 bit patterns (little-endian in the block)."""
    byte = code | code << 2 | code << 4 | code << 6
    blk = bytes([byte] * 8) + bytes([d_bits & 0xFF, d_bits >> 8, m_bits & 0xFF, m_bits >> 8])
    return np.frombuffer(blk * (n_rows * K // 32), np.uint8).copy()


def test_moe_tolerance_hand_worked_element(orc):
    """One expert, H = F = 32, every weight 1 (code 1, d = 1, m = 0), x = e_0, zero router
    logits (g = 1).  Then gate_f = up_f = 1, h_f = silu(1) = sigma(1), the gate and up bounds are
    2e-3 * 1, and for every output n:
      tol = 2e-3 * 32 * sigma(1) + 32 * 2e-3 * (silu'(1) * 1 + silu(1) * 1)
          = 0.064 * (2 sigma(1) + silu'(1)),
    with sigma(1) = 0.7310585786300049 and silu'(1) = sigma(1) + sigma(1)(1 - sigma(1))
    = 0.9276705118714868, i.e. tol = 0.064 * 2.3897876691314966 = 0.1529464108244158.
    Y_n = 32 * sigma(1) = 23.393874516160157."""
    H = F = 32
    one = _q2b32_constant_rows(F, H, 1, 0x3C00)
    X = np.zeros((1, H), np.uint16)
    X[0, 0] = 0x3F80  # bf16 1.0
    out = orc.moe(one, one, one, 1, H, F, 1, X, np.zeros((1, 1), np.float32))
    np.testing.assert_allclose(out["Y"][0], np.full(H, 23.393874516160157), rtol=1e-14)
    np.testing.assert_allclose(out["tol"][0], np.full(H, 0.1529464108244158), rtol=1e-13)


def test_pq_verify_accept_threshold_is_p_over_q(orc):
    """Accept iff u < p(x)/q(x): the largest fp32 below the ratio accepts, the smallest fp32
    at or above it rejects (the ratio taken from scipy's softmax, not the oracle)."""
    rng = np.random.default_rng(41)
    V, k, T = 12, 3, 0.9
    for trial in range(30):
        tl = rng.normal(0, 1.5, size=(1, k + 1, V)).astype(np.float32)
        dl = (tl[:, :k] + rng.normal(0, 1, size=(1, k, V))).astype(np.float32)
        x = rng.integers(0, V, size=(1, k)).astype(np.int32)
        p = _softmax_rows(tl[0], T)
        q = _softmax_rows(dl[0], T)
        for i in range(k):
            r = p[i, x[0, i]] / q[i, x[0, i]]
            if r >= 1:
                continue
            u = np.zeros((1, k), np.float32)      # rows before i accept (u = 0 < r)
            below = np.nextafter(np.float32(r), np.float32(0))
            if float(below) >= r:
                below = np.nextafter(below, np.float32(0))
            above = np.float32(r)
            if float(above) < r:
                above = np.nextafter(above, np.float32(1))
            u[0, i] = below
            out = orc.pq_verify(tl, dl, x, u, np.array([0.5], np.float32), T)
            assert out["n_acc"][0] > i
            u[0, i] = above
            out = orc.pq_verify(tl, dl, x, u, np.array([0.5], np.float32), T)
            assert out["n_acc"][0] == i


def test_pq_verify_strict_comparison_at_zero_ratio(orc):
    """p(x) = 0 exactly and u = 0: u < p/q is false, so the draft is rejected (a non-strict
    comparison would accept a token the target never emits)."""
    V, k = 6, 1
    tl = np.zeros((1, 2, V), np.float32)
    tl[0, 0, 2] = -1e4            # exp underflows: p_0(2) == 0 exactly
    dl = np.zeros((1, 1, V), np.float32)
    out = orc.pq_verify(tl, dl, np.array([[2]], np.int32), np.array([[0.0]], np.float32),
                        np.array([0.25], np.float32), 1.0)
    assert out["n_acc"][0] == 0 and out["tokens"][0, 0] != 2


# ---------------------------------------------------------------- greedy and per-session T

def _greedy_case(seed, S=6, k=4, V=40):
    """Logits on a 0.5 grid (distinct values, gaps >= 0.5) and drafts that are the argmax of
    their draft logits, which agree with the target argmax for a random prefix."""
    rng = np.random.default_rng(seed)
    t = np.stack([np.stack([rng.permutation(V) * 0.5 for _ in range(k + 1)]) for _ in range(S)]).astype(np.float32)
    d = np.stack([np.stack([rng.permutation(V) * 0.5 for _ in range(k)]) for _ in range(S)]).astype(np.float32)
    for s in range(S):
        agree = rng.integers(0, k + 1)
        for i in range(agree):
            d[s, i] = t[s, i]
    x = np.argmax(d, axis=2).astype(np.int32)
    ua = rng.random((S, k)).astype(np.float32)
    uf = rng.random(S).astype(np.float32)
    return t, d, x, ua, uf


def test_greedy_is_the_zero_temperature_limit(orc):
    """At T = 1e-4 every softmax of these logits is exactly one-hot in fp64 (the next value is
    5000 nats down), so the sampling verify must emit the greedy verify's tokens."""
    for seed in range(5):
        t, d, x, ua, uf = _greedy_case(seed)
        S = t.shape[0]
        g = orc.pq_verify(t, d, x, ua, uf, 1.0, temps=np.zeros(S), want_probs=True)
        sm = orc.pq_verify(t, d, x, ua, uf, 1e-4, want_probs=True)
        assert np.array_equal(g["n_acc"], sm["n_acc"]) and np.array_equal(g["tokens"], sm["tokens"])
        assert np.array_equal(g["probs"], sm["probs"])  # one-hot rows both ways
        assert np.all(g["fin_src"] == 3)
        assert 0 < g["n_acc"].min() or g["n_acc"].max() > 0  # the cases accept something


def test_greedy_ties_go_to_the_lower_index(orc):
    V, k = 8, 2
    t = np.zeros((1, k + 1, V), np.float32)
    t[0, 0, [2, 5]] = 3.0     # tie: argmax is 2
    t[0, 1, [1, 6]] = 1.0     # tie: argmax is 1
    t[0, 2, :] = -1.0         # all equal: argmax is 0
    d = np.zeros((1, k, V), np.float32)
    g = orc.pq_verify(t, d, np.array([[2, 6]], np.int32), np.zeros((1, k), np.float32),
                      np.zeros(1, np.float32), 1.0, temps=np.zeros(1))
    assert g["n_acc"][0] == 1 and list(g["tokens"][0]) == [2, 1, -1]
    g = orc.pq_verify(t, d, np.array([[2, 1]], np.int32), np.zeros((1, k), np.float32),
                      np.zeros(1, np.float32), 1.0, temps=np.zeros(1))
    assert g["n_acc"][0] == 2 and list(g["tokens"][0]) == [2, 1, 0]


def test_per_session_temperature_matches_the_scalar_verify(orc):
    st = synth.streams(0)
    S, k, V = 6, 4, 256
    v = synth.verify_inputs(st, S, k, V, 2.0, 0.5, 1.0)
    temps = np.array([0.5, 1.0, 2.0, 0.0, 0.7, 1.0])
    got = orc.pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], 1.0, temps=temps,
                        want_probs=True)
    for s in range(S):
        sl = slice(s, s + 1)
        if temps[s] > 0:
            ref = orc.pq_verify(v["target"][sl], v["draft"][sl], v["drafts"][sl], v["u_acc"][sl], v["u_fin"][sl],
                                float(temps[s]), want_probs=True)
        else:
            ref = orc.pq_verify(v["target"][sl], v["draft"][sl], v["drafts"][sl], v["u_acc"][sl], v["u_fin"][sl],
                                1.0, temps=np.zeros(1), want_probs=True)
        assert got["n_acc"][s] == ref["n_acc"][0]
        assert np.array_equal(got["tokens"][s], ref["tokens"][0])
        assert np.array_equal(got["probs"][s], ref["probs"][0])


def test_bad_temperature_marks_only_its_session(orc):
    st = synth.streams(0)
    S, k, V = 4, 3, 64
    v = synth.verify_inputs(st, S, k, V, 2.0, 0.5, 1.0)
    temps = np.array([1.0, -0.5, np.nan, 1.0])
    got = orc.pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], 1.0, temps=temps)
    assert got["bad_temperature"] and not got["bad_token"]
    assert list(got["n_acc"][1:3]) == [-1, -1] and np.all(got["tokens"][1:3] == -1)
    ref = orc.pq_verify(v["target"], v["draft"], v["drafts"], v["u_acc"], v["u_fin"], 1.0)
    assert np.array_equal(got["tokens"][[0, 3]], ref["tokens"][[0, 3]])
