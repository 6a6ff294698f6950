"""q2_tiny_gemm on the GPU against the fp64 oracle, element by element:
|gpu - oracle| <= 2e-3 * sum_k |a_k w_k|."""
import numpy as np
import pytest

from _util import check_gemm, to_dev
from speculative_decode_verifier_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(orc):
    import torch

    from speculative_decode_verifier_gb300 import build, q2v
    build.build()
    q2v.load()
    return torch.device("cuda:0"), q2v, orc


def _run(env, W, N, K, A, ws=None):
    dev, q2v, _ = env
    Y = q2v.q2_tiny_gemm(to_dev(W.reshape(-1), dev), N, K, to_dev(A, dev), ws=ws)
    return Y.cpu().numpy()


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_tiny_smoke_config(env, M):
    g = synth.config_gemm(0, M=M)
    Y = _run(env, g["W"], g["N"], g["K"], g["A"])
    Yo, absY = env[2].gemm(g["W"], g["N"], g["K"], g["A"])
    check_gemm(Y, Yo, absY, f"cfg0 M={M}")


def test_verifier_linear_config(env):
    g = synth.config_gemm(1)
    Y = _run(env, g["W"], g["N"], g["K"], g["A"])
    Yo, absY = env[2].gemm(g["W"], g["N"], g["K"], g["A"])
    worst = check_gemm(Y, Yo, absY, "cfg1")
    assert worst < 1e-4  # far inside the bound


@pytest.mark.parametrize("M,N,K", [
    (5, 517, 96),      # ragged N (not a multiple of 16), odd block count (3 blocks)
    (3, 33, 160),      # 5 blocks: a partial tile, 4-byte-aligned rows
    (7, 48, 288),      # 9 blocks: two tiles, the second nearly empty
    (8, 64, 4096),
    (9, 64, 1024),     # two activation slices
    (16, 40, 2048),
    (33, 50, 512),
    (64, 32, 4096),    # the largest M
    (5, 64, 8192),     # the largest K (32 warp tiles)
    (1, 1, 32),        # the smallest problem
    (6, 4100, 4064),   # a ragged last 16-row group at the verifier width; 127 blocks (odd), a partial 16th tile
    (8, 4864, 1024),   # 8 rows in one activation slice, 304 row groups
    (5, 12288, 4096),  # Q, K and V of the verifier layer as one linear (768 CTAs: two waves)
    (2, 38912, 512),   # the streaming kernel at every other row count: masked MMA columns
    (3, 38912, 512),
    (4, 38912, 512),
    (6, 38912, 512),
    (7, 38928, 512),   # and a unit count that is not a multiple of the SMs
    (5, 40960, 4096),  # the streaming kernel (many weight rows per SM): one session against a head
    (1, 65536, 256),   # streaming, one activation row, one K tile
    (8, 40000, 1024),  # streaming, all 8 columns of the MMA, units not a multiple of the warps
    (5, 40960, 8192),  # streaming at the largest K (the staged rows and the rings fill shared memory)
    (8, 39936, 8192),  # 8 rows at the largest K do not fit: the other kernels take it
])
def test_shapes(env, M, N, K):
    st = synth.Streams(1000 + M * 7 + N + K)
    W = synth.q2b32_weights(st, N, K)
    A = synth.activations_bf16(st, M, K)
    Y = _run(env, W, N, K, A)
    Yo, absY = env[2].gemm(W, N, K, A)
    check_gemm(Y, Yo, absY, f"M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(32, 512), (38912, 256)])  # per-CTA kernel; streaming kernel
def test_activation_range_extremes(env, N, K):
    """Rows far outside the f16 range, tiny rows and an all-zero row: the per-row power-of-two
    scale keeps them exact."""
    st = synth.Streams(77)
    M = 5
    W = synth.q2b32_weights(st, N, K)
    a = st["A"].normal(0, 1, size=(M, K))
    a[0] *= 1e30
    a[1] *= 1e-30
    a[2] = 0.0
    a[3] *= 7e4
    A = synth.bf16_bits(a)
    Y = _run(env, W, N, K, A)
    Yo, absY = env[2].gemm(W, N, K, A)
    assert np.all(Y[2] == 0.0)
    check_gemm(Y[[0, 1, 3, 4]], Yo[[0, 1, 3, 4]], absY[[0, 1, 3, 4]], "extremes")


@pytest.mark.parametrize("N", [48, 38912])  # per-CTA kernel; streaming kernel
def test_scale_extremes_within_range(env, N):
    """d = 0 (offset only), subnormal-small and the largest in-range scales."""
    st = synth.Streams(78)
    M, K = 4, 256
    codes = st["codes"].integers(0, 4, size=(N, K), dtype=np.uint8)
    d = st["d"].uniform(0.01, 0.05, size=(N, K // 32))
    d[0:16] = 0.0
    d[16:32] = 1e-6
    d[32:48] = 60.0    # the largest in-range scales (|d| < 64)
    m = st["m"].normal(0, 0.02, size=(N, K // 32))
    W = synth.pack_q2b32(codes, synth.fp16_bits(d), synth.fp16_bits(m))
    A = synth.activations_bf16(st, M, K)
    Y = _run(env, W, N, K, A)
    Yo, absY = env[2].gemm(W, N, K, A)
    check_gemm(Y, Yo, absY, "scales")


@pytest.mark.parametrize("N,K,row", [(16, 64, 3), (38912, 256, 38900)])  # per-CTA kernel; streaming kernel
def test_scale_out_of_range_sets_status(env, N, K, row):
    dev, q2v, _ = env
    st = synth.Streams(79)
    M = 2 if N < 1000 else 5
    codes = st["codes"].integers(0, 4, size=(N, K), dtype=np.uint8)
    d = np.full((N, K // 32), 0.02)
    d[row, 1] = 64.0
    W = synth.pack_q2b32(codes, synth.fp16_bits(d), synth.fp16_bits(np.zeros((N, K // 32))))
    A = synth.activations_bf16(st, M, K)
    ws = q2v.workspace(q2v.q2_tiny_gemm_workspace(M, N, K), dev)
    _run(env, W, N, K, A, ws=ws)
    assert q2v.q2_get_device_status(ws) == 8  # Q2_ERR_RANGE
    assert q2v.q2_get_device_status(ws) == 0  # read clears it


@pytest.mark.parametrize("N,K", [(4096, 4096), (40960, 4096)])  # per-CTA kernel; streaming kernel
def test_deterministic_and_ldy(env, N, K):
    """Repeated calls give the same bits (the streaming kernel sums the pieces of units cut between
    warps in warp order), and a padded output (ldy > N) keeps its padding."""
    import torch
    dev, q2v, orc = env
    g = synth.config_gemm(1, M=5, N=N, K=K)
    Wd = to_dev(g["W"].reshape(-1), dev)
    Ad = to_dev(g["A"], dev)
    Y1 = q2v.q2_tiny_gemm(Wd, g["N"], g["K"], Ad).cpu()
    Y2 = q2v.q2_tiny_gemm(Wd, g["N"], g["K"], Ad).cpu()
    assert torch.equal(Y1, Y2)
    # a padded output (ldy > N) leaves the padding untouched
    Yp = torch.full((5, g["N"] + 8), 7.0, device=dev)
    q2v.q2_tiny_gemm(Wd, g["N"], g["K"], Ad, Y=Yp)
    assert torch.equal(Yp[:, :g["N"]].cpu(), Y1)
    assert torch.all(Yp[:, g["N"]:] == 7.0)


def test_probe_brackets_the_gemm_kernel(env):
    """q2_set_probe records the caller's events around the GEMM kernel alone."""
    import torch
    dev, q2v, _ = env
    g = synth.config_gemm(1, M=5)
    Wd = to_dev(g["W"].reshape(-1), dev)
    Ad = to_dev(g["A"], dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    b.record()
    q2v.q2_set_probe(q2v.PROBE_GEMM, a, b)
    try:
        q2v.q2_tiny_gemm(Wd, g["N"], g["K"], Ad)
    finally:
        q2v.q2_set_probe(q2v.PROBE_NONE)
    torch.cuda.synchronize()
    assert 0.0 < a.elapsed_time(b) < 100.0
    with pytest.raises(q2v.Q2Error):
        q2v.q2_set_probe(99, a, b)
    with pytest.raises(q2v.Q2Error):
        q2v.q2_set_probe(q2v.PROBE_GEMM, None, None)


# ---- the tcgen05 path: K % 128 == 0 and 17 <= M <= 64, or 5 <= M <= 16 with enough 128-row
# tiles per SM (on a 152-SM GB300: N >= 32,832 at 5..8 rows, N >= 16,416 at 9..16 rows);
# other shapes take mma.sync

@pytest.mark.parametrize("M,N,K", [
    (17, 129, 128),     # one stage, ragged N just past one 128-row tile, 32-row padding
    (24, 300, 256),
    (32, 128, 4096),    # exactly one tile
    (33, 1, 128),       # a single output row (the rest of the tile is TMA zero fill)
    (40, 257, 1024),    # 48-row padding
    (48, 1000, 512),
    (60, 2049, 4096),   # the cohort row count, many tiles per CTA, ragged tail
    (64, 4096, 8192),   # the largest M and K
    (20, 127, 384),     # three stages, fewer rows than a tile
    (24, 100000, 256),  # 782 tiles: 5-6 per CTA, a full group of 4 then a partial one
    (48, 160000, 128),  # 1250 tiles: 8-9 per CTA, two full groups and a one-tile group
    (33, 50, 160),      # K % 128 != 0: the mma.sync path
    (5, 33000, 256),    # 5 rows, enough tiles per SM: tcgen05 with 16-column padding, ragged tail
    (8, 40000, 128),    # 8 rows, one stage
    (9, 16500, 512),    # 9 rows
    (16, 20000, 384),   # 16 rows, three stages
    (4, 50000, 256),    # 4 rows: stays on mma.sync however many weight rows
])
def test_umma_shapes(env, M, N, K):
    st = synth.Streams(5000 + M * 7 + N + K)
    W = synth.q2b32_weights(st, N, K)
    A = synth.activations_bf16(st, M, K)
    Y = _run(env, W, N, K, A)
    Yo, absY = env[2].gemm(W, N, K, A)
    check_gemm(Y, Yo, absY, f"M={M} N={N} K={K}")


def test_umma_activation_and_scale_extremes(env):
    """Per-row exponents far apart within one tile, a zero row, and the largest in-range
    scales, on the tcgen05 path."""
    st = synth.Streams(81)
    M, N, K = 24, 200, 512
    codes = st["codes"].integers(0, 4, size=(N, K), dtype=np.uint8)
    d = st["d"].uniform(0.01, 0.05, size=(N, K // 32))
    d[0:16] = 0.0
    d[16:40] = 60.0
    m = st["m"].normal(0, 0.02, size=(N, K // 32))
    W = synth.pack_q2b32(codes, synth.fp16_bits(d), synth.fp16_bits(m))
    a = st["A"].normal(0, 1, size=(M, K))
    a[0] *= 1e30
    a[1] *= 1e-30
    a[2] = 0.0
    a[3] *= 7e4
    A = synth.bf16_bits(a)
    Y = _run(env, W, N, K, A)
    Yo, absY = env[2].gemm(W, N, K, A)
    assert np.all(Y[2] == 0.0)
    rows = [r for r in range(M) if r != 2]
    check_gemm(Y[rows], Yo[rows], absY[rows], "umma extremes")


def test_umma_scale_out_of_range_sets_status(env):
    dev, q2v, _ = env
    st = synth.Streams(82)
    N, K, M = 160, 256, 20
    codes = st["codes"].integers(0, 4, size=(N, K), dtype=np.uint8)
    d = np.full((N, K // 32), 0.02)
    d[150, 5] = -64.0
    W = synth.pack_q2b32(codes, synth.fp16_bits(d), synth.fp16_bits(np.zeros((N, K // 32))))
    A = synth.activations_bf16(st, M, K)
    ws = q2v.workspace(q2v.q2_tiny_gemm_workspace(M, N, K), dev)
    _run(env, W, N, K, A, ws=ws)
    assert q2v.q2_get_device_status(ws) == 8  # Q2_ERR_RANGE
    assert q2v.q2_get_device_status(ws) == 0


def test_umma_deterministic_and_ldy(env):
    import torch
    dev, q2v, _ = env
    st = synth.Streams(83)
    M, N, K = 60, 700, 1024
    W = synth.q2b32_weights(st, N, K)
    A = synth.activations_bf16(st, M, K)
    Wd, Ad = to_dev(W.reshape(-1), dev), to_dev(A, dev)
    Y1 = q2v.q2_tiny_gemm(Wd, N, K, Ad).cpu()
    Y2 = q2v.q2_tiny_gemm(Wd, N, K, Ad).cpu()
    assert torch.equal(Y1, Y2)
    Yp = torch.full((M, N + 5), 7.0, device=dev)
    q2v.q2_tiny_gemm(Wd, N, K, Ad, Y=Yp)
    assert torch.equal(Yp[:, :N].cpu(), Y1)
    assert torch.all(Yp[:, N:] == 7.0)


def test_activation_magnitude_varies_along_k(env):
    """One power-of-two scale per activation row: slices of one row 1e20 apart, and a row that is
    zero in some slices only, stay within the bound."""
    st = synth.Streams(78)
    M, N, K = 5, 48, 4096
    W = synth.q2b32_weights(st, N, K)
    a = st["A"].normal(0, 1, size=(M, K))
    a[0, :256] *= 1e20
    a[1, 1024:2048] = 0.0
    a[2, ::2] *= 1e-20
    A = synth.bf16_bits(a)
    Y = _run(env, W, N, K, A)
    Yo, absY = env[2].gemm(W, N, K, A)
    check_gemm(Y, Yo, absY, "magnitudes along K")
