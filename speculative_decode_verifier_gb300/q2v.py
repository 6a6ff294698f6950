"""Thin ctypes binding of libq2v (the C ABI declared in include/q2v.h).

Argument marshalling only: each function checks dtype/device/contiguity of the torch
tensors it is given, passes their device pointers and the current CUDA stream to the C
entry point of the same name, and raises on a non-OK status.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback of any kind, and a
missing library is an error.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libq2v.so")

Q2_OK = 0
STATUS_NAMES = {0: "Q2_OK", 1: "Q2_ERR_INVALID_ARG", 2: "Q2_ERR_ALIGNMENT", 3: "Q2_ERR_UNSUPPORTED",
                4: "Q2_ERR_WORKSPACE", 5: "Q2_ERR_CUDA", 6: "Q2_ERR_TIMEOUT", 7: "Q2_ERR_BAD_TOKEN",
                8: "Q2_ERR_RANGE", 9: "Q2_ERR_BAD_TEMPERATURE"}
MOE_RENORMALIZE = 1
LM_HEAD_FUSE_STATS = 1
EXPORTS = ("q2_tiny_gemm_workspace", "q2_tiny_gemm", "q2_moe_grouped_workspace", "q2_moe_grouped",
           "pq_verify_workspace", "pq_verify", "pq_verify_noalloc", "q2_get_device_status", "q2_status_string",
           "q2_version", "q2_set_probe", "pq_verify_ex", "q2_quench_init", "q2_quench_update",
           "q2_lm_head_verify_workspace", "q2_lm_head_verify", "q2_selftest_wait_timeout",
           "q2_hbm_read_probe")

# kernels that q2_set_probe can bracket (q2_probe_kernel)
PROBE_NONE, PROBE_MOE_GATE_UP, PROBE_MOE_DOWN, PROBE_GEMM, PROBE_PQ_STATS, PROBE_PQ_VERIFY = range(6)


class Q2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libq2v.so (build it first with speculative_decode_verifier_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libq2v.so is not built ({path}); run `python -c \"import __graft_entry__ as g; "
                           f"g.build()\"` first")
    lib = ctypes.CDLL(path)
    P, I, U, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_float, ctypes.c_size_t
    lib.q2_tiny_gemm_workspace.argtypes = [I, I, I]
    lib.q2_tiny_gemm_workspace.restype = Z
    lib.q2_tiny_gemm.argtypes = [P, I, I, P, I, I, P, I, P, Z, P]
    lib.q2_tiny_gemm.restype = I
    lib.q2_moe_grouped_workspace.argtypes = [I, I, I, I, I]
    lib.q2_moe_grouped_workspace.restype = Z
    lib.q2_moe_grouped.argtypes = [P, P, P, I, I, I, I, U, P, I, P, P, P, P, P, Z, P]
    lib.q2_moe_grouped.restype = I
    lib.pq_verify_workspace.argtypes = [I, I, I]
    lib.pq_verify_workspace.restype = Z
    lib.pq_verify.argtypes = [P, P, P, P, P, I, I, I, F, P, P, P, P, Z, P]
    lib.pq_verify.restype = I
    lib.pq_verify_ex.argtypes = [P, P, P, P, P, I, I, I, P, P, P, P, P, Z, P]
    lib.pq_verify_ex.restype = I
    lib.pq_verify_noalloc.argtypes = [P, P, P, P, P, I, I, I, F, P, P, P, P]
    lib.pq_verify_noalloc.restype = I
    lib.q2_get_device_status.argtypes = [P, P]
    lib.q2_get_device_status.restype = I
    lib.q2_status_string.argtypes = [I]
    lib.q2_status_string.restype = ctypes.c_char_p
    lib.q2_version.restype = I
    lib.q2_lm_head_verify_workspace.argtypes = [I, I, I, I]
    lib.q2_lm_head_verify_workspace.restype = Z
    lib.q2_lm_head_verify.argtypes = [P, I, I, P, I, P, P, P, P, I, I, P, F, U, P, P, P, P, P, Z, P]
    lib.q2_lm_head_verify.restype = I
    lib.q2_quench_init.argtypes = [P, I]
    lib.q2_quench_init.restype = I
    lib.q2_quench_update.argtypes = [P, I, P, ctypes.c_double, ctypes.c_double]
    lib.q2_quench_update.restype = I
    lib.q2_set_probe.argtypes = [I, P, P]
    lib.q2_set_probe.restype = I
    lib.q2_selftest_wait_timeout.argtypes = [P, Z, P]
    lib.q2_selftest_wait_timeout.restype = I
    lib.q2_hbm_read_probe.argtypes = [P, Z, P, P]
    lib.q2_hbm_read_probe.restype = I
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().q2_status_string(int(status)).decode()


def version() -> int:
    return load().q2_version()


def q2_status_string(status: int) -> str:
    return status_string(status)


def q2_version() -> int:
    return version()


class QuenchState(ctypes.Structure):
    """q2_quench_state: the running regret, the steps counted, quenched (0/1)."""
    _fields_ = [("regret", ctypes.c_double), ("steps", ctypes.c_int), ("quenched", ctypes.c_int)]


QUENCH_GUARD = 2.16      # plain steps per verify step (the pages' calibration)
QUENCH_THRESHOLD = 4.0   # plain-step deficit that quenches a request


def q2_quench_init(S: int):
    """A fresh q2_quench_state array of S sessions (host memory)."""
    state = (QuenchState * S)()
    _raise(load().q2_quench_init(state, S), "q2_quench_init")
    return state


def q2_quench_update(state, n_accepted, guard: float = 2.16, threshold: float = 4.0) -> int:
    """One verify step over len(state) sessions; returns the number newly quenched."""
    import numpy as np
    a = np.ascontiguousarray(np.asarray(n_accepted, dtype=np.int32))
    if a.shape != (len(state),):
        raise ValueError(f"n_accepted must have shape ({len(state)},)")
    r = load().q2_quench_update(state, len(state), a.ctypes.data_as(ctypes.c_void_p), float(guard), float(threshold))
    if r < 0:
        raise Q2Error(1, "q2_quench_update")
    return r


class YieldQuench:
    """Host-side yield-quench controller for S sessions (state kept in the library's C struct)."""

    def __init__(self, S: int, guard: float = QUENCH_GUARD, threshold: float = QUENCH_THRESHOLD):
        self.S, self.guard, self.threshold = S, float(guard), float(threshold)
        self.state = q2_quench_init(S)

    def update(self, n_accepted) -> int:
        """One verify step; n_accepted: int32 host array [S] (a torch CPU tensor or numpy).
        Returns the number of sessions this step quenched."""
        return q2_quench_update(self.state, n_accepted, self.guard, self.threshold)

    def quenched(self):
        return [bool(self.state[s].quenched) for s in range(self.S)]

    def regret(self):
        return [self.state[s].regret for s in range(self.S)]


def q2_set_probe(kernel: int, ev_begin=None, ev_end=None) -> None:
    """Bracket every later launch of `kernel` (a PROBE_* id) with the two torch.cuda.Event
    records; PROBE_NONE turns the hook off.  The events must be created with timing."""
    b = None if ev_begin is None else ctypes.c_void_p(ev_begin.cuda_event)
    e = None if ev_end is None else ctypes.c_void_p(ev_end.cuda_event)
    _raise(load().q2_set_probe(int(kernel), b, e), "q2_set_probe")


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t: torch.Tensor | None, name: str, dtype, nullable: bool = False):
    if t is None:
        if nullable:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _raise(st: int, where: str):
    if st != Q2_OK:
        raise Q2Error(st, where)


# ------------------------------------------------------------------ workspaces

def q2_tiny_gemm_workspace(M: int, N: int, K: int) -> int:
    return load().q2_tiny_gemm_workspace(M, N, K)


def q2_moe_grouped_workspace(M: int, E: int, topk: int, H: int, F: int) -> int:
    return load().q2_moe_grouped_workspace(M, E, topk, H, F)


def pq_verify_workspace(S: int, k: int, V: int) -> int:
    return load().pq_verify_workspace(S, k, V)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed device workspace (uint8) of at least nbytes, 256-byte aligned."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def q2_get_device_status(ws: torch.Tensor, stream=None) -> int:
    return load().q2_get_device_status(_ptr(ws), ctypes.c_void_p(_stream(stream)))


def q2_selftest_wait_timeout(ws: torch.Tensor, stream=None) -> None:
    """Launch the failure-detection self-test: a bounded device wait that nothing completes
    records Q2_ERR_TIMEOUT in ws's status word after 1 s (read it with q2_get_device_status)."""
    _check(ws, "ws", torch.uint8)
    _raise(load().q2_selftest_wait_timeout(_ptr(ws), ws.numel(), ctypes.c_void_p(_stream(stream))),
           "q2_selftest_wait_timeout")


# ------------------------------------------------------------------ entry points

def q2_hbm_read_probe(buf: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """Enqueue one read of every byte of `buf` (a contiguous CUDA tensor whose byte size is a
    multiple of 16) on the current stream; `sink` is a CUDA int32/uint32 tensor of >= 1 element."""
    _check(buf, "buf", buf.dtype if isinstance(buf, torch.Tensor) else None)
    _check(sink, "sink", torch.int32)
    nbytes = buf.numel() * buf.element_size()
    _raise(load().q2_hbm_read_probe(_ptr(buf), nbytes, _ptr(sink), _stream(stream)), "q2_hbm_read_probe")


def q2_tiny_gemm(W: torch.Tensor, N: int, K: int, A: torch.Tensor, Y: torch.Tensor | None = None,
                 ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = A W^T.  W: uint8 Q2B32 bytes of an [N,K] matrix; A: bf16 [M,K] (int16/uint16 bit
    patterns or torch.bfloat16); Y: fp32 [M,N] (allocated if None)."""
    _check(W, "W", torch.uint8)
    if A.dtype == torch.bfloat16:
        A = A.view(torch.int16)
    _check(A, "A", torch.int16)
    M = A.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(Y, "Y", torch.float32)
    if ws is None:
        ws = workspace(q2_tiny_gemm_workspace(M, N, K), A.device)
    st = load().q2_tiny_gemm(_ptr(W), N, K, _ptr(A), M, A.shape[1], _ptr(Y), Y.shape[1], _ptr(ws),
                             ws.numel(), ctypes.c_void_p(_stream(stream)))
    _raise(st, "q2_tiny_gemm")
    return Y


def q2_moe_grouped(Wg, Wu, Wd, E: int, H: int, F: int, topk: int, X: torch.Tensor, router: torch.Tensor,
                   Y: torch.Tensor | None = None, ids_out: torch.Tensor | None = None,
                   w_out: torch.Tensor | None = None, renormalize: bool = False,
                   ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    for t, n in ((Wg, "Wg"), (Wu, "Wu"), (Wd, "Wd")):
        _check(t, n, torch.uint8)
    if X.dtype == torch.bfloat16:
        X = X.view(torch.int16)
    _check(X, "X", torch.int16)
    _check(router, "router", torch.float32)
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, H), dtype=torch.float32, device=X.device)
    _check(Y, "Y", torch.float32)
    _check(ids_out, "ids_out", torch.int32, nullable=True)
    _check(w_out, "w_out", torch.float32, nullable=True)
    if ws is None:
        ws = workspace(q2_moe_grouped_workspace(M, E, topk, H, F), X.device)
    st = load().q2_moe_grouped(_ptr(Wg), _ptr(Wu), _ptr(Wd), E, H, F, topk,
                               MOE_RENORMALIZE if renormalize else 0, _ptr(X), M, _ptr(router), _ptr(Y),
                               _ptr(ids_out), _ptr(w_out), _ptr(ws), ws.numel(),
                               ctypes.c_void_p(_stream(stream)))
    _raise(st, "q2_moe_grouped")
    return Y


def pq_verify(target: torch.Tensor, draft: torch.Tensor | None, drafts: torch.Tensor | None,
              u_acc: torch.Tensor | None, u_fin: torch.Tensor, temperature: float,
              n_acc: torch.Tensor | None = None, tokens: torch.Tensor | None = None,
              probs: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """Returns (n_acc [S] int32, tokens [S,k+1] int32).  target [S,k+1,V] fp32, draft [S,k,V]
    fp32, drafts [S,k] int32, u_acc [S,k] fp32, u_fin [S] fp32."""
    _check(target, "target", torch.float32)
    S, k1, V = target.shape
    k = k1 - 1
    if k > 0:
        _check(draft, "draft", torch.float32)
        _check(drafts, "drafts", torch.int32)
        _check(u_acc, "u_acc", torch.float32)
    _check(u_fin, "u_fin", torch.float32)
    dev = target.device
    if n_acc is None:
        n_acc = torch.empty(S, dtype=torch.int32, device=dev)
    if tokens is None:
        tokens = torch.empty((S, k + 1), dtype=torch.int32, device=dev)
    _check(n_acc, "n_acc", torch.int32)
    _check(tokens, "tokens", torch.int32)
    _check(probs, "probs", torch.float32, nullable=True)
    if ws is None:
        ws = workspace(pq_verify_workspace(S, k, V), dev)
    st = load().pq_verify(_ptr(target), _ptr(draft) if k > 0 else None, _ptr(drafts) if k > 0 else None,
                          _ptr(u_acc) if k > 0 else None, _ptr(u_fin), S, k, V, float(temperature),
                          _ptr(n_acc), _ptr(tokens), _ptr(probs), _ptr(ws), ws.numel(),
                          ctypes.c_void_p(_stream(stream)))
    _raise(st, "pq_verify")
    return n_acc, tokens


def pq_verify_ex(target: torch.Tensor, draft: torch.Tensor | None, drafts: torch.Tensor | None,
                 u_acc: torch.Tensor | None, u_fin: torch.Tensor, temperatures: torch.Tensor,
                 n_acc: torch.Tensor | None = None, tokens: torch.Tensor | None = None,
                 probs: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """pq_verify with one temperature per session (fp32 [S] on the device; 0 = the greedy
    verify).  Returns (n_acc [S] int32, tokens [S,k+1] int32)."""
    _check(target, "target", torch.float32)
    S, k1, V = target.shape
    k = k1 - 1
    if k > 0:
        _check(draft, "draft", torch.float32)
        _check(drafts, "drafts", torch.int32)
        _check(u_acc, "u_acc", torch.float32)
    _check(u_fin, "u_fin", torch.float32)
    _check(temperatures, "temperatures", torch.float32)
    dev = target.device
    if n_acc is None:
        n_acc = torch.empty(S, dtype=torch.int32, device=dev)
    if tokens is None:
        tokens = torch.empty((S, k + 1), dtype=torch.int32, device=dev)
    _check(n_acc, "n_acc", torch.int32)
    _check(tokens, "tokens", torch.int32)
    _check(probs, "probs", torch.float32, nullable=True)
    if ws is None:
        ws = workspace(pq_verify_workspace(S, k, V), dev)
    st = load().pq_verify_ex(_ptr(target), _ptr(draft) if k > 0 else None, _ptr(drafts) if k > 0 else None,
                             _ptr(u_acc) if k > 0 else None, _ptr(u_fin), S, k, V, _ptr(temperatures),
                             _ptr(n_acc), _ptr(tokens), _ptr(probs), _ptr(ws), ws.numel(),
                             ctypes.c_void_p(_stream(stream)))
    _raise(st, "pq_verify_ex")
    return n_acc, tokens


def q2_lm_head_verify_workspace(S: int, k: int, V: int, K: int) -> int:
    return load().q2_lm_head_verify_workspace(S, k, V, K)


def q2_lm_head_verify(W: torch.Tensor, V: int, K: int, A: torch.Tensor, draft: torch.Tensor | None,
                      drafts: torch.Tensor | None, u_acc: torch.Tensor | None, u_fin: torch.Tensor,
                      S: int, k: int, temperatures: torch.Tensor | None = None, temperature: float = 1.0,
                      fuse_stats: bool = False, target: torch.Tensor | None = None, n_acc: torch.Tensor | None = None,
                      tokens: torch.Tensor | None = None, probs: torch.Tensor | None = None,
                      ws: torch.Tensor | None = None, stream=None):
    """Vocabulary head + verify: target = A W^T as [S, k+1, V] fp32, then the p/q verify over it
    (temperatures: fp32 [S] on the device, 0 = greedy; else one temperature).  Returns
    (target, n_acc, tokens)."""
    _check(W, "W", torch.uint8)
    if A.dtype == torch.bfloat16:
        A = A.view(torch.int16)
    _check(A, "A", torch.int16)
    if k > 0:
        _check(draft, "draft", torch.float32)
        _check(drafts, "drafts", torch.int32)
        _check(u_acc, "u_acc", torch.float32)
    _check(u_fin, "u_fin", torch.float32)
    _check(temperatures, "temperatures", torch.float32, nullable=True)
    dev = A.device
    if target is None:
        target = torch.empty((S, k + 1, V), dtype=torch.float32, device=dev)
    if n_acc is None:
        n_acc = torch.empty(S, dtype=torch.int32, device=dev)
    if tokens is None:
        tokens = torch.empty((S, k + 1), dtype=torch.int32, device=dev)
    for t, n in ((target, "target"),):
        _check(t, n, torch.float32)
    _check(n_acc, "n_acc", torch.int32)
    _check(tokens, "tokens", torch.int32)
    _check(probs, "probs", torch.float32, nullable=True)
    if ws is None:
        ws = workspace(q2_lm_head_verify_workspace(S, k, V, K), dev)
    st = load().q2_lm_head_verify(_ptr(W), V, K, _ptr(A), A.shape[1], _ptr(draft) if k > 0 else None,
                                  _ptr(drafts) if k > 0 else None, _ptr(u_acc) if k > 0 else None, _ptr(u_fin),
                                  S, k, _ptr(temperatures), float(temperature), LM_HEAD_FUSE_STATS if fuse_stats else 0,
                                  _ptr(target), _ptr(n_acc),
                                  _ptr(tokens), _ptr(probs), _ptr(ws), ws.numel(), ctypes.c_void_p(_stream(stream)))
    _raise(st, "q2_lm_head_verify")
    return target, n_acc, tokens


def pq_verify_noalloc(target: torch.Tensor, draft: torch.Tensor | None, drafts: torch.Tensor | None,
                      u_acc: torch.Tensor | None, u_fin: torch.Tensor, temperature: float,
                      n_acc: torch.Tensor, tokens: torch.Tensor, probs: torch.Tensor | None = None,
                      stream=None):
    """pq_verify with the library's fixed scratch instead of a workspace, for callers that
    cannot allocate device memory.  The caller provides every output tensor (nothing is
    allocated here either).  Returns (n_acc, tokens)."""
    _check(target, "target", torch.float32)
    S, k1, V = target.shape
    k = k1 - 1
    if k > 0:
        _check(draft, "draft", torch.float32)
        _check(drafts, "drafts", torch.int32)
        _check(u_acc, "u_acc", torch.float32)
    _check(u_fin, "u_fin", torch.float32)
    _check(n_acc, "n_acc", torch.int32)
    _check(tokens, "tokens", torch.int32)
    _check(probs, "probs", torch.float32, nullable=True)
    st = load().pq_verify_noalloc(_ptr(target), _ptr(draft) if k > 0 else None, _ptr(drafts) if k > 0 else None,
                                  _ptr(u_acc) if k > 0 else None, _ptr(u_fin), S, k, V, float(temperature),
                                  _ptr(n_acc), _ptr(tokens), _ptr(probs), ctypes.c_void_p(_stream(stream)))
    _raise(st, "pq_verify_noalloc")
    return n_acc, tokens
