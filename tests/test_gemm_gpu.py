"""f16_gemm (TMA + tcgen05) on the GPU against the oracle's binary64 GEMM."""
import numpy as np
import pytest

import oracle
import synth
from _gpu import require_gpu, to_dev, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    require_gpu()
    import int4_weight_only_affine_gb300 as w4
    return w4


@pytest.mark.parametrize("M,N,K", [
    (1, 8, 8), (3, 24, 40), (128, 256, 64), (130, 264, 200), (257, 520, 1000),
    (200, 1000, 896), (64, 2048, 128), (300, 256, 4096),
])
def test_gemm_small_full_compare(w4, M, N, K):
    x = synth.make_half_matrix(M + N, M, K)
    w = synth.make_half_matrix(K + 7, K, N, std=0.05)
    y = w4.f16_gemm(to_dev(x), to_dev(w)).cpu().numpy()
    yo, ad = oracle.gemm(x, w, M, N, K)
    ok, worst = within_tol(y, yo, ad)
    assert ok, f"worst err/tol = {worst}"
    assert w4.device_status() == 0


# Every output of the CTA-pair kernel at the prefill lengths, with ragged
# column tiles (N = 2040, 520) and ragged row tiles (M = 1570, 300); K = 64
# keeps the full oracle comparison quick.
@pytest.mark.parametrize("M,N", [(1570, 2040), (512, 11008), (4096, 2560), (300, 520), (1570, 2560)])
def test_gemm_pair_full_compare(w4, M, N):
    K = 64
    x = synth.make_half_matrix(51 + M, M, K)
    w = synth.make_half_matrix(52 + N, K, N, std=0.05)
    y = w4.f16_gemm(to_dev(x), to_dev(w)).cpu().numpy()
    yo, ad = oracle.gemm(x, w, M, N, K)
    ok, worst = within_tol(y, yo, ad)
    assert ok, f"worst err/tol = {worst}"
    assert w4.device_status() == 0


def _entries(M, N, n=1500, seed=0):
    g = np.random.default_rng(seed)
    ms = g.integers(0, M, size=n)
    ns = g.integers(0, N, size=n)
    # rows at the edges of the 128- and 256-row tiles, including the first row
    # of a ragged last tile
    split = (M // 256) * 256
    edge_m = [0, M - 1, min(M - 1, 127), min(M - 1, 128), max(0, split - 1), min(M - 1, split)]
    edge_n = [0, N - 1, min(N - 1, 255), min(N - 1, 256)]
    ms = np.concatenate([ms, np.repeat(edge_m, len(edge_n))])
    ns = np.concatenate([ns, np.tile(edge_n, len(edge_m))])
    return ms.astype(np.int32), ns.astype(np.int32)


@pytest.mark.parametrize("K,N", sorted({(K, N) for _, K, N in synth.QWEN25_3B}))
@pytest.mark.parametrize("M", [1570])
def test_gemm_prefill_shapes_sampled(w4, M, K, N):
    x = synth.make_half_matrix(11 + K, M, K)
    w = synth.make_half_matrix(12 + N, K, N, std=0.05)
    y = w4.f16_gemm(to_dev(x), to_dev(w)).cpu().numpy()
    ms, ns = _entries(M, N)
    yo, ad = oracle.gemm_entries(x, w, N, K, ms, ns)
    ok, worst = within_tol(y[ms, ns], yo, ad)
    assert ok, f"worst err/tol = {worst}"
    assert w4.device_status() == 0


@pytest.mark.parametrize("M", [128, 512, 4096])
def test_gemm_other_prefill_lengths(w4, M):
    K, N = 2048, 11008
    x = synth.make_half_matrix(21 + M, M, K)
    w = synth.make_half_matrix(22, K, N, std=0.05)
    y = w4.f16_gemm(to_dev(x), to_dev(w)).cpu().numpy()
    ms, ns = _entries(M, N, n=800)
    yo, ad = oracle.gemm_entries(x, w, N, K, ms, ns)
    ok, worst = within_tol(y[ms, ns], yo, ad)
    assert ok, f"worst err/tol = {worst}"


def test_dequant_then_gemm_equals_gemv(w4):
    """Invariant of the prefill path: GEMM on the dequantised scratch agrees with
    the fused GEMV (both against the oracle's fused result)."""
    M, N, K = 4, 2048, 2048
    qw, s, b = synth.make_linear(31, N, K)
    x = synth.make_x(32, M, K)
    tq, ts, tb, tx = to_dev(qw), to_dev(s), to_dev(b), to_dev(x)
    yg = w4.f16_gemm(tx, w4.w4_dequant_f16(tq, ts, tb)).cpu().numpy()
    yv = w4.w4_gemv(tx, tq, ts, tb).cpu().numpy()
    yo, ad = oracle.gemv(x, qw, s, b, N, K, threads=8)
    assert within_tol(yg, yo, ad)[0] and within_tol(yv, yo, ad)[0]


def test_gemm_row_tail_keeps_stream_order(w4):
    """A GEMM reading the previous GEMM's output right after it (no
    synchronisation, M = 1570 with a ragged 256-row tile) sees all of it:
    bit-identical to the same chain with a synchronisation in between (the
    kernels are deterministic)."""
    import torch
    M, K, N = 1570, 1024, 1024
    x = to_dev(synth.make_half_matrix(31, M, K))
    w1 = to_dev(synth.make_half_matrix(32, K, N, std=0.05))
    w2 = to_dev(synth.make_half_matrix(33, N, N, std=0.05))
    y1 = w4.f16_gemm(x, w1)
    y2 = w4.f16_gemm(y1, w2)
    torch.cuda.synchronize()
    z1 = w4.f16_gemm(x, w1)
    torch.cuda.synchronize()
    z2 = w4.f16_gemm(z1, w2)
    torch.cuda.synchronize()
    assert torch.equal(y1, z1)
    assert torch.equal(y2, z2)
    assert w4.device_status() == 0


@pytest.mark.parametrize("M", [100, 1570])
def test_gemm_overlap_flag_keeps_dependencies(w4, M):
    """With OVERLAP_PREVIOUS a GEMM fetches its weights early but reads x and
    writes y only after the previous kernel: a read-after-write chain (x is
    the previous output) and a write-after-read (y is the previous kernel's
    input) give the same bits as with synchronisations in between."""
    import torch
    K, N = 1024, 1024
    x = to_dev(synth.make_half_matrix(41, M, K))
    w1 = to_dev(synth.make_half_matrix(42, K, N, std=0.05))
    w2 = to_dev(synth.make_half_matrix(43, N, N, std=0.05))
    ov = w4.OVERLAP_PREVIOUS
    # reference, synchronised
    r1 = w4.f16_gemm(x, w1); torch.cuda.synchronize()
    r2 = w4.f16_gemm(r1, w2); torch.cuda.synchronize()
    r3 = w4.f16_gemm(r2, w2); torch.cuda.synchronize()
    # overlapped: y1 -> y2 (RAW), then y3 = f(y2) written into y1's buffer while
    # the GEMM before it read y1 (WAR), then one more read of it
    y1 = w4.f16_gemm(x, w1)
    y2 = w4.f16_gemm(y1, w2, flags=ov)
    w4.f16_gemm(y2, w2, y=y1, flags=ov)
    torch.cuda.synchronize()
    assert torch.equal(y2, r2)
    assert torch.equal(y1, r3)
    assert w4.device_status() == 0
