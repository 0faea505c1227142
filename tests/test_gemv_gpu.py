"""w4_gemv on the GPU against the CPU oracle (tolerance 1e-3 * sum|w x| + 1e-3)."""
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


SMALL = [
    (1, 896, 896),     # single GEMV of the 0.5B q projection
    (1, 1000, 896),
    (1, 1, 64),        # one row, one group
    (16, 1, 64),
    (2, 257, 128),     # ragged row tail
    (3, 33, 64),
    (8, 130, 640),
    (9, 77, 192),      # second activation tile, partially filled
    (16, 300, 1024),
    (4, 2048, 2048),   # cluster split along K
    (1, 256, 2048),
    (5, 1000, 3072),
    (16, 1024, 1024),
]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_gemv_matches_oracle(w4, M, N, K):
    qw, s, b = synth.make_linear(1000 + N + K, N, K)
    x = synth.make_x(7 + M, M, K)
    y = w4.w4_gemv(to_dev(x), to_dev(qw), to_dev(s), to_dev(b)).cpu().numpy()
    yo, ad = oracle.gemv(x, qw, s, b, N, K, threads=8)
    ok, worst = within_tol(y, yo, ad)
    assert ok, f"worst err/tol = {worst}"


def _sample_rows(N, n=96, seed=0):
    g = np.random.default_rng(seed)
    fixed = [0, 1, 15, 16, N // 2, N - 17, N - 16, N - 1]
    rows = np.unique(np.concatenate([[r for r in fixed if 0 <= r < N], g.integers(0, N, size=n)]))
    return rows.astype(np.int32)


FULL = sorted({(K, N) for _, K, N in synth.QWEN25_3B + synth.QWEN3_06B})


@pytest.mark.parametrize("K,N", FULL)
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_gemv_full_size_sampled_rows(w4, M, K, N):
    qw, s, b = synth.make_linear(synth.layer_seed(2000, 0, N % 7), N, K)
    x = synth.make_x(3000 + M, M, K)
    y = w4.w4_gemv(to_dev(x), to_dev(qw), to_dev(s), to_dev(b)).cpu().numpy()
    rows = _sample_rows(N, n=48 if M > 4 else 96)
    yo, ad = oracle.gemv_rows(x, qw, s, b, K, rows)
    ok, worst = within_tol(y[:, rows], yo, ad)
    assert ok, f"worst err/tol = {worst}"


def test_gemv_deterministic_and_zero_cases(w4):
    import torch
    M, N, K = 3, 2048, 11008
    qw, s, b = synth.make_linear(77, N, K)
    x = synth.make_x(78, M, K)
    args = (to_dev(x), to_dev(qw), to_dev(s), to_dev(b))
    y1 = w4.w4_gemv(*args)
    y2 = w4.w4_gemv(*args)
    assert torch.equal(y1, y2)
    # Codes 8 with bias -8*scale make every weight exactly zero: sum_k |w x| = 0,
    # so the tolerance is the absolute 1e-3 (the folded scale and bias terms
    # cancel up to fp32 rounding).
    z = w4.w4_gemv(args[0], to_dev(np.full_like(qw, 0x88888888)), args[2],
                   to_dev((-8.0 * s.astype(np.float64)).astype(np.float16)))
    assert torch.max(torch.abs(z.float())).item() <= 1e-3


def test_gemv_closed_form_q8_zero_bias(w4):
    """All q = 8, bias = 0, integer activations: y = 8 * sum_g scale_g * sum_{k in g} x_k."""
    M, N, K = 4, 96, 1024
    g = np.random.default_rng(5)
    qw = np.full((N, K // 8), 0x88888888, dtype=np.uint32)
    s, _ = synth.make_scales_biases(g, N, K)
    b = np.zeros_like(s)
    x = g.integers(-3, 4, size=(M, K)).astype(np.float16)
    y = w4.w4_gemv(to_dev(x), to_dev(qw), to_dev(s), to_dev(b)).cpu().numpy().astype(np.float64)
    xs = x.astype(np.float64).reshape(M, K // 64, 64).sum(axis=2)          # [M][groups]
    want = 8.0 * xs @ s.astype(np.float64).T
    assert np.all(np.abs(y - want) <= 1e-3 * np.abs(want) + 1e-3)
