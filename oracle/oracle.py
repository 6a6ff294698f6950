"""Python access to the fp64 CPU oracle (``q2v_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path (the CUDA library and its
binding) never imports this module; the two share no code.

Each wrapper takes plain numpy arrays (the bit patterns of bf16/fp16 tensors as
uint16, fp32 logits as float32, Q2B32 weights as uint8 bytes) and returns fp64
results.  The C source documents the definitions and the readings it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q2v_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libq2v_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc -O2 (no fast-math) and OpenMP; return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, f64 = ctypes.c_int, ctypes.c_double
        lib.orc_half_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_half_to_f64.restype = f64
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = f64
        lib.orc_q2b32_dequant.argtypes = [P, i32, i32, P]
        lib.orc_gemm.argtypes = [P, i32, i32, P, i32, i32, P, P, i32]
        lib.orc_softmax.argtypes = [P, i32, f64, P]
        lib.orc_inverse_cdf.argtypes = [P, i32, f64, P, P]
        lib.orc_inverse_cdf.restype = i32
        lib.orc_pq_verify.argtypes = [P, P, P, P, P, i32, i32, i32, f64,
                                      P, P, P, P, P, P, P, i32]
        lib.orc_pq_verify.restype = i32
        lib.orc_pq_verify_ex.argtypes = [P, P, P, P, P, i32, i32, i32, f64, P,
                                         P, P, P, P, P, P, P, i32]
        lib.orc_pq_verify_ex.restype = i32
        lib.orc_moe.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, i32, P, P, P, P, P, i32]
        lib.orc_version.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def half_to_f64(bits: int) -> float:
    return _load().orc_half_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return _load().orc_bf16_to_f64(int(bits))


def dequant(W: np.ndarray, N: int, K: int) -> np.ndarray:
    """Q2B32 bytes of an [N,K] matrix -> fp64 [N,K]."""
    W = _c(W, np.uint8)
    assert K % 32 == 0 and W.size == N * (K // 32) * 12
    out = np.empty((N, K), np.float64)
    _load().orc_q2b32_dequant(_ptr(W), N, K, _ptr(out))
    return out


def gemm(W: np.ndarray, N: int, K: int, A_bits: np.ndarray, threads: int | None = None):
    """Y = A W^T in fp64 and absY = sum_k |a w|.  A_bits: bf16 bit patterns [M,K]."""
    W = _c(W, np.uint8)
    A = _c(A_bits, np.uint16)
    M = A.shape[0]
    assert A.shape[1] >= K
    Y = np.empty((M, N), np.float64)
    absY = np.empty((M, N), np.float64)
    _load().orc_gemm(_ptr(W), N, K, _ptr(A), M, A.shape[1], _ptr(Y), _ptr(absY),
                     threads or default_threads())
    return Y, absY


def softmax(x: np.ndarray, T: float = 1.0) -> np.ndarray:
    x = _c(x, np.float32)
    p = np.empty(x.shape[-1], np.float64)
    _load().orc_softmax(_ptr(x), x.shape[-1], float(T), _ptr(p))
    return p


def inverse_cdf(w: np.ndarray, u: float):
    """(y, cell_lo, cell_hi) for the smallest y with C(y) > u*Z."""
    w = _c(w, np.float64)
    lo = np.zeros(1, np.float64)
    hi = np.zeros(1, np.float64)
    y = _load().orc_inverse_cdf(_ptr(w), w.size, float(u), _ptr(lo), _ptr(hi))
    return y, float(lo[0]), float(hi[0])


def pq_verify(target, draft, drafts, u_acc, u_fin, T: float, want_probs: bool = False,
              threads: int | None = None, temps=None) -> dict:
    """The p/q verify for S sessions.  target [S,k+1,V] fp32, draft [S,k,V] fp32,
    drafts [S,k] int32, u_acc [S,k] fp32, u_fin [S] fp32.  temps: optional [S] per-session
    temperatures (0 = the greedy verify); T is used for every session when it is None."""
    target = _c(target, np.float32)
    S, k1, V = target.shape
    k = k1 - 1
    draft = _c(draft, np.float32).reshape(S, k, V) if k > 0 else np.zeros((S, 0, V), np.float32)
    drafts = _c(drafts, np.int32).reshape(S, k)
    u_acc = _c(u_acc, np.float32).reshape(S, k)
    u_fin = _c(u_fin, np.float32).reshape(S)
    n_acc = np.empty(S, np.int32)
    tokens = np.empty((S, k + 1), np.int32)
    probs = np.empty((S, 2 * k + 1, V), np.float64) if want_probs else None
    ratio = np.empty((S, k), np.float64)
    lo = np.empty(S, np.float64)
    hi = np.empty(S, np.float64)
    src = np.empty(S, np.int32)
    tv = None if temps is None else _c(temps, np.float64).reshape(S)
    bad = _load().orc_pq_verify_ex(_ptr(target), _ptr(draft), _ptr(drafts), _ptr(u_acc), _ptr(u_fin),
                                   S, k, V, float(T), _ptr(tv), _ptr(n_acc), _ptr(tokens), _ptr(probs),
                                   _ptr(ratio), _ptr(lo), _ptr(hi), _ptr(src),
                                   threads or default_threads())
    return dict(n_acc=n_acc, tokens=tokens, probs=probs, ratio=ratio, cell_lo=lo, cell_hi=hi,
                fin_src=src, bad_token=bool(bad & 1), bad_temperature=bool(bad & 2))


def moe(Wg, Wu, Wd, E: int, H: int, F: int, topk: int, X_bits, router, renorm: bool = False,
        threads: int | None = None) -> dict:
    """Routed MoE FFN; returns Y [M,H] fp64, ids, weights and the parity bound tol [M,H]."""
    Wg, Wu, Wd = _c(Wg, np.uint8), _c(Wu, np.uint8), _c(Wd, np.uint8)
    X = _c(X_bits, np.uint16)
    router = _c(router, np.float32)
    M = X.shape[0]
    assert X.shape[1] == H and router.shape == (M, E)
    Y = np.empty((M, H), np.float64)
    ids = np.empty((M, topk), np.int32)
    gw = np.empty((M, topk), np.float64)
    tol = np.empty((M, H), np.float64)
    _load().orc_moe(_ptr(Wg), _ptr(Wu), _ptr(Wd), E, H, F, topk, int(bool(renorm)), _ptr(X), M,
                    _ptr(router), _ptr(Y), _ptr(ids), _ptr(gw), _ptr(tol),
                    threads or default_threads())
    return dict(Y=Y, ids=ids, weights=gw, tol=tol)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
