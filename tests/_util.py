"""Shared helpers of the parity tests: moving seeded inputs to the device and comparing the
CUDA path with the oracle under the stated acceptance rules."""
from __future__ import annotations

import os
import re
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent.parent

# GEMM: |gpu - oracle| <= 2e-3 * sum_k |a_k w_k| per element.
GEMM_REL = 2e-3
# probabilities: within 1e-5 absolute.
PROB_ATOL = 1e-5
# a uniform within this of a decision boundary (p/q, or a normalised CDF cell edge) is a
# near-tie: the token may differ there, and such draws are counted and reported.
NEAR_TIE = 1e-5

# every compare_verify result of this test session, as (test id, counts); conftest.py prints
# the per-test totals at the end of the run and writes them to $Q2V_NEAR_TIE_REPORT when set
NEAR_TIE_LOG: list[tuple[str, dict]] = []


def header_functions() -> list[str]:
    """Names of the functions include/q2v.h declares."""
    text = (ROOT / "include" / "q2v.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def to_dev(a: np.ndarray, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


def check_gemm(Y_gpu: np.ndarray, Y_orc: np.ndarray, absY: np.ndarray, what: str = "") -> float:
    err = np.abs(Y_gpu.astype(np.float64) - Y_orc)
    bound = GEMM_REL * absY
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} elements over 2e-3*sum|a w|; worst ratio "
                           f"{np.max(err / np.maximum(absY, 1e-300))}")
    return float(np.max(err / np.maximum(absY, 1e-300)))


def _cells(w: np.ndarray):
    c = np.cumsum(w)
    Z = c[-1]
    return np.concatenate([[0.0], c[:-1]]) / Z, c / Z


def compare_verify(gpu_n, gpu_tok, orc: dict, u_acc, u_fin, k: int) -> dict:
    """Token-level parity.  Outside near-ties the GPU result must equal the oracle's.
    At a near-tie the GPU result must still be one the exact arithmetic reaches for some
    uniform within NEAR_TIE of the given one.  Returns counts."""
    gpu_n = np.asarray(gpu_n)
    gpu_tok = np.asarray(gpu_tok)
    S = gpu_n.shape[0]
    probs = orc["probs"]
    stats = dict(sessions=S, exact=0, accept_near_ties=0, draw_near_ties=0, mismatches_at_near_ties=0)
    for s in range(S):
        jo = int(orc["n_acc"][s])
        jg = int(gpu_n[s])
        same = jg == jo and np.array_equal(gpu_tok[s], orc["tokens"][s])
        # near-ties among the accept decisions the oracle evaluated
        acc_tie = False
        for i in range(min(jo + 1, k)):
            r = orc["ratio"][s, i]
            if np.isfinite(r) and abs(float(u_acc[s, i]) - r) < NEAR_TIE:
                acc_tie = True
        u = float(u_fin[s])
        draw_tie = (abs(u - orc["cell_lo"][s]) < NEAR_TIE) or (abs(u - orc["cell_hi"][s]) < NEAR_TIE)
        stats["accept_near_ties"] += int(acc_tie)
        stats["draw_near_ties"] += int(draw_tie)
        if same:
            stats["exact"] += 1
            continue
        assert acc_tie or draw_tie, (f"session {s}: gpu n_acc={jg} tokens={gpu_tok[s].tolist()} vs oracle "
                                     f"n_acc={jo} tokens={orc['tokens'][s].tolist()} with no near-tie")
        stats["mismatches_at_near_ties"] += 1
        if jg == jo and probs is not None:
            # same accept path: the GPU's final token must own a cell within NEAR_TIE of u
            assert np.array_equal(gpu_tok[s, :jg], orc["tokens"][s, :jo])
            y = int(gpu_tok[s, jg])
            if jo < k:
                w = np.maximum(probs[s, jo] - probs[s, k + 1 + jo], 0.0)
                if w.sum() == 0:
                    w = probs[s, jo]
            else:
                w = probs[s, k]
            lo, hi = _cells(w)
            assert w[y] > 0 and lo[y] - NEAR_TIE <= u <= hi[y] + NEAR_TIE, (s, y, lo[y], hi[y], u)
    NEAR_TIE_LOG.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], dict(stats)))
    return stats
