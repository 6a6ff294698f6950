"""pq_verify_noalloc: the verify for callers that cannot allocate device memory (for example
a decode loop inside a framework whose pool owns the device).  It must give exactly what
pq_verify gives with a caller-provided workspace, on consecutive calls that reuse its fixed
scratch, and refuse sizes the scratch cannot hold.  This file runs last so that a failure here
leaves every other result already reported."""
import ctypes

import numpy as np
import pytest

from _util import to_dev
from speculative_decode_verifier_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    return torch.device("cuda:0"), q2v, q2v.load()


def _call_noalloc_c(lib, t, S, k, V, T, n_acc, toks, stream):
    """Through the C ABI directly: device pointers, sizes, the stream."""
    P = ctypes.c_void_p
    return lib.pq_verify_noalloc(P(t["target"].data_ptr()), P(t["draft"].data_ptr()), P(t["drafts"].data_ptr()),
                                 P(t["u_acc"].data_ptr()), P(t["u_fin"].data_ptr()), S, k, V, float(T),
                                 P(n_acc.data_ptr()), P(toks.data_ptr()), None, P(stream))


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(env):
    import torch
    dev, q2v, lib = env
    stream = torch.cuda.current_stream().cuda_stream
    for salt in (0, 1):  # two calls in a row on the shared scratch, different inputs
        v = synth.config_verify(3, salt=salt)
        S, k1, V = v["target"].shape
        t = {n: to_dev(v[n], dev) for n in ("target", "draft", "drafts", "u_acc", "u_fin")}
        n_ref, tok_ref = q2v.pq_verify(t["target"], t["draft"], t["drafts"], t["u_acc"], t["u_fin"], v["T"])
        n_acc = torch.full((S,), -7, dtype=torch.int32, device=dev)
        toks = torch.full((S, k1), -7, dtype=torch.int32, device=dev)
        assert _call_noalloc_c(lib, t, S, k1 - 1, V, v["T"], n_acc, toks, stream) == 0
        torch.cuda.synchronize()
        # same kernels and arithmetic: the results must agree exactly
        assert torch.equal(n_acc.cpu(), n_ref.cpu())
        assert torch.equal(toks.cpu(), tok_ref.cpu())


def test_noalloc_at_its_largest_size(env):
    """S = 15 sessions at k = 4, V = 129,280: the largest verify the 2 MiB scratch holds, run and
    compared with the workspace entry point."""
    import torch
    dev, q2v, lib = env
    assert q2v.pq_verify_workspace(15, 4, 129280) <= 2 << 20 < q2v.pq_verify_workspace(16, 4, 129280)
    stream = torch.cuda.current_stream().cuda_stream
    v = synth.verify_inputs(synth.Streams(4242), 15, 4, 129280, t_std=3.0, noise_std=1.0, T=1.0)
    S, k1, V = v["target"].shape
    t = {n: to_dev(v[n], dev) for n in ("target", "draft", "drafts", "u_acc", "u_fin")}
    n_ref, tok_ref = q2v.pq_verify(t["target"], t["draft"], t["drafts"], t["u_acc"], t["u_fin"], v["T"])
    n_acc = torch.full((S,), -7, dtype=torch.int32, device=dev)
    toks = torch.full((S, k1), -7, dtype=torch.int32, device=dev)
    assert _call_noalloc_c(lib, t, S, k1 - 1, V, v["T"], n_acc, toks, stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(n_acc.cpu(), n_ref.cpu())
    assert torch.equal(toks.cpu(), tok_ref.cpu())


def test_noalloc_binding_and_bad_token(env):
    import torch
    dev, q2v, lib = env
    v = synth.config_verify(3, salt=2)
    v["drafts"] = v["drafts"].copy()
    v["drafts"][1, 0] = v["target"].shape[2]  # out of range
    S, k1, V = v["target"].shape
    t = {n: to_dev(v[n], dev) for n in ("target", "draft", "drafts", "u_acc", "u_fin")}
    n_acc = torch.empty(S, dtype=torch.int32, device=dev)
    toks = torch.empty((S, k1), dtype=torch.int32, device=dev)
    q2v.pq_verify_noalloc(t["target"], t["draft"], t["drafts"], t["u_acc"], t["u_fin"], v["T"], n_acc, toks)
    n = n_acc.cpu().numpy()
    assert n[1] == -1 and np.all(toks.cpu().numpy()[1] == -1)
    n_ref, tok_ref = q2v.pq_verify(t["target"], t["draft"], t["drafts"], t["u_acc"], t["u_fin"], v["T"])
    assert np.array_equal(n, n_ref.cpu().numpy())


def test_noalloc_refuses_sizes_beyond_its_scratch(env):
    _, q2v, lib = env
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: the call is refused before anything is enqueued
    S, k, V = 4096, 16, 129280
    assert q2v.pq_verify_workspace(S, k, V) > (2 << 20)
    st = lib.pq_verify_noalloc(fake, fake, fake, fake, fake, S, k, V, 1.0, fake, fake, None, None)
    assert st == 3  # Q2_ERR_UNSUPPORTED


def _driver():
    """libcuda (the driver API) through ctypes: stream capture and graph node counts."""
    drv = ctypes.CDLL("libcuda.so.1")
    begin = getattr(drv, "cuStreamBeginCapture_v2", None) or drv.cuStreamBeginCapture
    begin.argtypes = [ctypes.c_void_p, ctypes.c_int]
    drv.cuStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    drv.cuGraphGetNodes.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)]
    drv.cuGraphDestroy.argtypes = [ctypes.c_void_p]
    return drv, begin


def test_noalloc_rejected_call_enqueues_nothing(env):
    """A call refused on the host (bad temperature, oversized S) adds no work to the stream: a
    capture around it yields a graph with no nodes."""
    import torch
    dev, q2v, lib = env
    drv, begin = _driver()
    s = torch.cuda.Stream(device=dev)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: both calls are refused on the host
    for S, T, want in ((2, -1.0, 1), (16, 1.0, 3)):
        assert begin(ctypes.c_void_p(s.cuda_stream), 2) == 0  # relaxed capture mode
        st = lib.pq_verify_noalloc(fake, fake, fake, fake, fake, S, 4, 129280, T, fake, fake, None,
                                   ctypes.c_void_p(s.cuda_stream))
        graph = ctypes.c_void_p()
        assert drv.cuStreamEndCapture(ctypes.c_void_p(s.cuda_stream), ctypes.byref(graph)) == 0
        n = ctypes.c_size_t(0)
        assert drv.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
        drv.cuGraphDestroy(graph)
        assert st == want
        assert n.value == 0
