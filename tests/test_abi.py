"""The C ABI without a GPU: the library builds, loads and exports every function that
include/q2v.h declares; workspace queries; host-side argument errors come back before
anything is enqueued (these calls never touch a device)."""
import ctypes
import subprocess

import pytest

from _util import ROOT, header_functions


@pytest.fixture(scope="module")
def lib():
    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    return q2v.load()


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("q2_tiny_gemm", "q2_tiny_gemm_workspace", "q2_moe_grouped", "q2_moe_grouped_workspace",
              "pq_verify", "pq_verify_workspace", "q2_get_device_status", "q2_status_string", "q2_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    from speculative_decode_verifier_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in header_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_binding_names_match_header():
    from speculative_decode_verifier_gb300 import q2v
    assert set(q2v.EXPORTS) == set(header_functions())
    for n in q2v.EXPORTS:
        assert callable(getattr(q2v, n)), n


def test_version_and_status_strings(lib):
    assert lib.q2_version() == 100
    for code in range(10):
        assert lib.q2_status_string(code)
    assert lib.q2_status_string(99) == b"unknown status"


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "q2v.h"\nint main(void){ return (int)q2_tiny_gemm_workspace(5,4096,4096) > 0 ? 0 : 1; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", str(src), "-I", str(ROOT / "include"),
                    "-o", str(tmp_path / "t.o")], check=True)


def test_workspace_queries(lib):
    # the prepared activations dominate the GEMM workspace; it fits either path, and the
    # tcgen05 operand pads M=5 to 16 columns
    g5 = lib.q2_tiny_gemm_workspace(5, 4096, 4096)
    assert 256 + 16 * 4096 * 2 <= g5 < 256 + 16 * 4096 * 4
    assert lib.q2_tiny_gemm_workspace(5, 129280, 4096) == g5   # the size does not depend on N
    assert lib.q2_tiny_gemm_workspace(3, 4096, 160) < 256 + 3 * 160 * 4 + 4096  # K % 128 != 0: mma.sync only
    assert lib.q2_tiny_gemm_workspace(60, 129280, 4096) >= 256 + 64 * 4096 * 2  # 60 rows pad to 64 columns
    assert lib.q2_tiny_gemm_workspace(0, 4096, 4096) == 256       # invalid sizes: header only
    assert lib.pq_verify_workspace(1, 4, 1024) == 256             # small-V tier needs only the header
    pq3 = lib.pq_verify_workspace(3, 4, 129280)
    assert pq3 >= 256 + 3 * 9 * 8 and pq3 < 4 << 20
    assert lib.pq_verify_workspace(3, 4, 129280) < lib.pq_verify_workspace(12, 4, 129280)
    assert lib.q2_moe_grouped_workspace(5, 64, 6, 4096, 2048) > 30 * 2048 * 8


P = ctypes.c_void_p
FAKE = P(1 << 20)            # 16-byte aligned, never dereferenced: these calls fail host-side
FAKE_MIS = P((1 << 20) + 4)


def _gemm(lib, W=FAKE, N=16, K=256, A=FAKE, M=2, lda=256, Y=FAKE, ldy=16, ws=FAKE, wsb=1 << 30):
    return lib.q2_tiny_gemm(W, N, K, A, M, lda, Y, ldy, ws, wsb, None)


def test_gemm_host_errors(lib):
    assert _gemm(lib, W=None) == 1
    assert _gemm(lib, N=0) == 1
    assert _gemm(lib, K=100) == 1
    assert _gemm(lib, K=0) == 1
    assert _gemm(lib, lda=128) == 1
    assert _gemm(lib, ldy=8) == 1
    assert _gemm(lib, M=0) == 1
    assert _gemm(lib, M=65) == 3
    assert _gemm(lib, K=8192 + 32, lda=8192 + 32) == 3
    assert _gemm(lib, W=FAKE_MIS) == 2
    assert _gemm(lib, A=FAKE_MIS) == 2
    assert _gemm(lib, lda=260) == 2
    assert _gemm(lib, ws=None) == 4
    assert _gemm(lib, wsb=100) == 4
    assert _gemm(lib, ws=FAKE_MIS) == 4


def _pq(lib, t=FAKE, d=FAKE, x=FAKE, ua=FAKE, uf=FAKE, S=2, k=4, V=8192, T=1.0, n=FAKE, tok=FAKE, pr=None,
        ws=FAKE, wsb=1 << 30):
    return lib.pq_verify(t, d, x, ua, uf, S, k, V, T, n, tok, pr, ws, wsb, None)


def test_pq_verify_host_errors(lib):
    assert _pq(lib, T=0.0) == 1
    assert _pq(lib, T=-1.0) == 1
    assert _pq(lib, T=float("inf")) == 1
    assert _pq(lib, T=float("nan")) == 1
    assert _pq(lib, S=0) == 1
    assert _pq(lib, V=0) == 1
    assert _pq(lib, k=-1) == 1
    assert _pq(lib, k=17) == 3
    assert _pq(lib, d=None) == 1
    assert _pq(lib, t=None) == 1
    assert _pq(lib, t=FAKE_MIS) == 2
    assert _pq(lib, d=FAKE_MIS) == 2
    assert _pq(lib, ws=None) == 4
    assert _pq(lib, wsb=300) == 4


def _moe(lib, E=8, H=256, F=128, topk=2, flags=0, M=5, ws=FAKE, wsb=1 << 30, X=FAKE):
    return lib.q2_moe_grouped(FAKE, FAKE, FAKE, E, H, F, topk, flags, X, M, FAKE, FAKE, None, None, ws, wsb,
                              None)


def test_moe_host_errors(lib):
    assert _moe(lib, topk=0) == 1
    assert _moe(lib, topk=9) == 1
    assert _moe(lib, H=100) == 1
    assert _moe(lib, flags=4) == 1
    assert _moe(lib, M=0) == 1
    assert _moe(lib, M=65) == 3
    assert _moe(lib, E=300, topk=2) == 3
    assert _moe(lib, X=FAKE_MIS) == 2
    assert _moe(lib, wsb=1000) == 4


def test_selftest_wait_timeout_host_errors(lib):
    # workspace checks come before any launch
    assert lib.q2_selftest_wait_timeout(None, 1 << 20, None) == 4
    assert lib.q2_selftest_wait_timeout(FAKE_MIS, 1 << 20, None) == 4
    assert lib.q2_selftest_wait_timeout(FAKE, 100, None) == 4


def test_python_binding_refuses_cpu_tensors():
    import torch

    from speculative_decode_verifier_gb300 import q2v
    with pytest.raises(ValueError):
        q2v.q2_tiny_gemm(torch.zeros(16, dtype=torch.uint8), 1, 32, torch.zeros((1, 32), dtype=torch.int16))


def _noalloc(lib, S=2, k=4, V=129280, T=1.0, t=FAKE):
    return lib.pq_verify_noalloc(t, FAKE, FAKE, FAKE, FAKE, S, k, V, T, FAKE, FAKE, None, None)


def test_noalloc_size_limit_and_host_errors(lib):
    """The no-workspace verify holds a 2 MiB scratch: at k = 4, V = 129,280 the largest S whose
    pq_verify workspace fits is 15; S = 16 is refused with Q2_ERR_UNSUPPORTED.  Argument errors come
    back as pq_verify's, and every refusal happens before anything is enqueued (no device is
    touched here)."""
    assert lib.pq_verify_workspace(15, 4, 129280) <= 2 << 20
    assert lib.pq_verify_workspace(16, 4, 129280) > 2 << 20
    assert _noalloc(lib, S=16) == 3
    assert _noalloc(lib, S=4096, k=16) == 3
    assert _noalloc(lib, T=-1.0) == 1
    assert _noalloc(lib, T=float("nan")) == 1
    assert _noalloc(lib, S=0) == 1
    assert _noalloc(lib, k=17) == 3
    assert _noalloc(lib, t=FAKE_MIS) == 2
