"""Seeded synthetic inputs for the verifier step (shared by the tests, the smoke check
and the benchmark).

This module holds none of the verifier's arithmetic: it only draws random numbers
and rounds them to their storage types.  Every tensor comes from numpy's PCG64,
seeded with ``SEED0 + config_id`` and split into one child stream per tensor in a
fixed order (``STREAMS``), so each tensor is reproducible on its own.

Workloads (the shapes and value laws of the five synthetic configurations):

* cfg0  tiny smoke: Q2B32 linear K=256, N=512, M=1..4; pq_verify S=1, k=4, V=1024,
        target logits ~ N(0, 2^2), draft = target + N(0, 0.5^2).
* cfg1  one verifier linear: K=N=4096, M=5 (1 committed + 4 draft rows).
* cfg2  routed MoE FFN: 64 experts, H=4096, F=2048, M=5, top-6, router ~ N(0,1).
* cfg3  batched pq_verify: S=3, k=4, V=129280, target ~ N(0, 3^2), draft = target + N(0,1), T=1.
* cfg4  cohort: M = 12 sessions x 5 rows = 60 rows against a K=4096, N=129280 lm_head,
        then pq_verify (S=12, k=4) over those logits with draft = logits + N(0,1).

Value laws shared by all weights: codes uniform on {0,1,2,3}; d ~ U(0.01, 0.05)
rounded to fp16; m ~ N(0, 0.02^2) rounded to fp16; activations ~ N(0,1) rounded to
bf16.  Uniforms for the verify are ``(bits32 >> 8) * 2^-24`` (exact fp32, in [0,1)).
Draft tokens stand in for the drafter: each x_i is drawn from softmax(draft_i / T)
by the Gumbel-max rule with its own seeded stream (a sampler unrelated to the
verify's inverse-CDF draws).
"""
from __future__ import annotations

import numpy as np

SEED0 = 20261202
STREAMS = ("codes", "d", "m", "A", "router", "t_logits", "noise", "draft_uniforms",
           "u_acc", "u_fin", "extra0", "extra1", "extra2", "extra3")

Q2B32_BLOCK_K = 32
Q2B32_BLOCK_BYTES = 12

CONFIGS = {
    0: dict(name="tiny smoke: Q2B32 linear K=256 N=512 M=1..4 + pq_verify S=1 k=4 V=1024",
            K=256, N=512, Ms=(1, 2, 3, 4), S=1, k=4, V=1024, t_std=2.0, noise_std=0.5, T=1.0),
    1: dict(name="verifier linear Q2B32 K=4096 N=4096 M=5", K=4096, N=4096, M=5),
    2: dict(name="MoE verifier FFN: 64 Q2B32 experts H=4096 F=2048 top-6 M=5",
            E=64, H=4096, F=2048, M=5, topk=6),
    3: dict(name="batched pq_verify S=3 k=4 V=129280 T=1", S=3, k=4, V=129280, t_std=3.0,
            noise_std=1.0, T=1.0),
    4: dict(name="cohort verify: M=60 (12x5) vs Q2B32 lm_head K=4096 N=129280, then pq_verify S=12 k=4",
            K=4096, N=129280, M=60, S=12, k=4, V=129280, noise_std=1.0, T=1.0),
}


class Streams:
    """One independent numpy Generator per named tensor, from one seed."""

    def __init__(self, seed: int):
        children = np.random.SeedSequence(seed).spawn(len(STREAMS))
        self._gens = {name: np.random.Generator(np.random.PCG64(c))
                      for name, c in zip(STREAMS, children)}

    def __getitem__(self, name: str) -> np.random.Generator:
        return self._gens[name]


def streams(config_id: int, salt: int = 0) -> Streams:
    return Streams(SEED0 + config_id + 1000 * salt)


# ----------------------------------------------------------------- rounding

def fp16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to IEEE binary16 (numpy's round-to-nearest-even); return bits."""
    return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to fp32 and then to bfloat16 (round-to-nearest-even at each step);
    return the 16-bit patterns."""
    f = np.ascontiguousarray(np.asarray(x, np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(f)
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact; a storage conversion)."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def uniforms_f32(g: np.random.Generator, shape) -> np.ndarray:
    """Uniforms (bits32 >> 8) * 2^-24: exactly representable in fp32, in [0, 1)."""
    bits = g.integers(0, 2 ** 32, size=shape, dtype=np.uint64)
    return ((bits >> np.uint64(8)).astype(np.float64) * 2.0 ** -24).astype(np.float32)


# ----------------------------------------------------------------- Q2B32 weights

def pack_q2b32(codes: np.ndarray, d_bits: np.ndarray, m_bits: np.ndarray) -> np.ndarray:
    """Pack codes [N,K] (values 0..3), fp16 scale/offset bits [N,K/32] into Q2B32 bytes
    [N, K/32, 12]: 8 code bytes (4 codes per byte, low bits first), d, m (little-endian)."""
    codes = np.asarray(codes, np.uint8)
    N, K = codes.shape
    nb = K // Q2B32_BLOCK_K
    c = codes.reshape(N, nb, 8, 4)
    packed = (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)
    out = np.empty((N, nb, Q2B32_BLOCK_BYTES), np.uint8)
    out[..., :8] = packed
    d = np.asarray(d_bits, np.uint16).reshape(N, nb)
    m = np.asarray(m_bits, np.uint16).reshape(N, nb)
    out[..., 8] = (d & 0xFF).astype(np.uint8)
    out[..., 9] = (d >> 8).astype(np.uint8)
    out[..., 10] = (m & 0xFF).astype(np.uint8)
    out[..., 11] = (m >> 8).astype(np.uint8)
    return out


def q2b32_weights(st: Streams, N: int, K: int, d_lo=0.01, d_hi=0.05, m_std=0.02,
                  batch: int = 1) -> np.ndarray:
    """Random Q2B32 weights for `batch` stacked [N,K] matrices, as uint8 bytes
    [batch*N, K/32, 12] (expert e's matrix is rows e*N..e*N+N-1)."""
    rows = batch * N
    nb = K // Q2B32_BLOCK_K
    out = np.empty((rows, nb, Q2B32_BLOCK_BYTES), np.uint8)
    # a uniform byte is four independent uniform 2-bit codes
    out[..., :8] = st["codes"].integers(0, 256, size=(rows, nb, 8), dtype=np.uint8)
    d = fp16_bits(st["d"].uniform(d_lo, d_hi, size=(rows, nb)))
    m = fp16_bits(st["m"].normal(0.0, m_std, size=(rows, nb)))
    out[..., 8:10] = d.view(np.uint8).reshape(rows, nb, 2)
    out[..., 10:12] = m.view(np.uint8).reshape(rows, nb, 2)
    return out


def activations_bf16(st: Streams, M: int, K: int, std: float = 1.0) -> np.ndarray:
    return bf16_bits(st["A"].normal(0.0, std, size=(M, K)))


# ----------------------------------------------------------------- verify inputs

def gumbel_max_drafts(draft_logits: np.ndarray, T: float, g: np.random.Generator) -> np.ndarray:
    """Stand-in drafter: x = argmax_v (draft[v]/T + G_v), G_v = -log(-log U_v), U_v in (0,1).
    This is the Gumbel-max sampler of softmax(draft/T); it is input generation only."""
    d = np.asarray(draft_logits, np.float64)
    U = g.random(size=d.shape)
    U = np.clip(U, 1e-300, 1.0 - 2.0 ** -53)
    G = -np.log(-np.log(U))
    return np.argmax(d / T + G, axis=-1).astype(np.int32)


def verify_inputs(st: Streams, S: int, k: int, V: int, t_std: float, noise_std: float, T: float,
                  target: np.ndarray | None = None) -> dict:
    """target [S,k+1,V] fp32 (drawn ~N(0,t_std^2) unless given), draft = target[:, :k] +
    N(0, noise_std^2) in fp32, drafts by Gumbel-max, u_acc [S,k], u_fin [S]."""
    if target is None:
        target = st["t_logits"].normal(0.0, t_std, size=(S, k + 1, V)).astype(np.float32)
    else:
        target = np.ascontiguousarray(target, np.float32).reshape(S, k + 1, V)
    noise = st["noise"].normal(0.0, noise_std, size=(S, k, V))
    draft = (target[:, :k, :].astype(np.float64) + noise).astype(np.float32)
    drafts = gumbel_max_drafts(draft, T, st["draft_uniforms"]) if k > 0 else np.zeros((S, 0), np.int32)
    u_acc = uniforms_f32(st["u_acc"], (S, k))
    u_fin = uniforms_f32(st["u_fin"], (S,))
    return dict(target=target, draft=np.ascontiguousarray(draft), drafts=drafts, u_acc=u_acc,
                u_fin=u_fin, T=float(T))


def config_gemm(config_id: int, M: int | None = None, N: int | None = None, K: int | None = None,
                salt: int = 0) -> dict:
    cfg = CONFIGS[config_id]
    st = streams(config_id, salt)
    N = N or cfg["N"]
    K = K or cfg["K"]
    M = M or cfg.get("M") or max(cfg["Ms"])
    return dict(W=q2b32_weights(st, N, K), A=activations_bf16(st, M, K), N=N, K=K, M=M)


def config_moe(config_id: int = 2, salt: int = 0, **over) -> dict:
    cfg = dict(CONFIGS[config_id])
    cfg.update(over)
    st = streams(config_id, salt)
    E, H, F, M, topk = cfg["E"], cfg["H"], cfg["F"], cfg["M"], cfg["topk"]
    Wg = q2b32_weights(st, F, H, batch=E)
    Wu = q2b32_weights(st, F, H, batch=E)
    Wd = q2b32_weights(st, H, F, batch=E)
    X = activations_bf16(st, M, H)
    router = st["router"].normal(0.0, 1.0, size=(M, E)).astype(np.float32)
    return dict(Wg=Wg, Wu=Wu, Wd=Wd, X=X, router=router, E=E, H=H, F=F, M=M, topk=topk)


def config_verify(config_id: int, salt: int = 0, **over) -> dict:
    cfg = dict(CONFIGS[config_id])
    cfg.update(over)
    st = streams(config_id, salt)
    return verify_inputs(st, cfg["S"], cfg["k"], cfg["V"], cfg["t_std"], cfg["noise_std"], cfg["T"])
