"""w4_dequant_f16 on the GPU: bit-exact against the oracle (binary16 RNE)."""
import numpy as np
import pytest

import oracle
import synth
from _gpu import require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    require_gpu()
    import int4_weight_only_affine_gb300 as w4
    return w4


def _dq(w4, qw, s, b):
    return w4.w4_dequant_f16(to_dev(qw), to_dev(s), to_dev(b)).cpu().numpy().view(np.uint16)


# N % 8 == 0 takes the tensor-copy kernel (tiles of 64 rows x 256 k, ragged in
# both directions here, several tiles per CTA for the largest), other N the
# shared-memory transpose kernel.
@pytest.mark.parametrize("N,K", [(1000, 896), (257, 192), (1, 64), (64, 64), (130, 128), (8, 640), (3, 1024),
                                 (4104, 2240), (136, 64)])
def test_dequant_bit_exact_small(w4, N, K):
    qw, s, b = synth.make_linear(10 + N + K, N, K)
    got = _dq(w4, qw, s, b)
    assert got.shape == (K, N)
    assert np.array_equal(got, oracle.dequant_f16_t(qw, s, b, N, K))


def test_dequant_bit_exact_extreme_values(w4):
    """Scales and biases drawn from every binary16 exponent (subnormals, overflow
    to infinity, exact cancellation to +-0) and every code."""
    g = np.random.default_rng(99)
    N, K = 512, 256

    def rnd_half(n):
        e = g.integers(0, 31, size=n)
        f = g.integers(0, 1024, size=n)
        sg = g.integers(0, 2, size=n)
        return ((sg << 15) | (e << 10) | f).astype(np.uint16)

    qw = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    s = rnd_half(N * K // 64).reshape(N, K // 64).view(np.float16)
    b = rnd_half(N * K // 64).reshape(N, K // 64).view(np.float16)
    s[0, 0] = np.float16(1.0)
    b[0, 0] = np.float16(-0.0)
    got = _dq(w4, qw, s, b)
    assert np.array_equal(got, oracle.dequant_f16_t(qw, s, b, N, K))


@pytest.mark.parametrize("K,N", sorted({(K, N) for _, K, N in synth.QWEN25_3B}))
def test_dequant_full_size_sampled(w4, K, N):
    qw, s, b = synth.make_linear(4000 + N, N, K)
    got = _dq(w4, qw, s, b)
    g = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, N - 1, N // 2], g.integers(0, N, size=40)])).astype(np.int32)
    want = oracle.dequant_f16_rows(qw, s, b, K, rows)
    assert np.array_equal(got[:, rows].T, want)


def test_dequant_independent_calls_overlap(w4):
    """Back-to-back calls into distinct scratch buffers with OVERLAP_PREVIOUS
    (each may run concurrently with the previous one) stay bit-exact."""
    import torch
    shapes = [(2560, 2048), (2048, 2048), (4104, 2240), (2048, 1024), (1000, 896)]
    mats = [synth.make_linear(7000 + i, N, K) for i, (N, K) in enumerate(shapes)]
    dev = [tuple(to_dev(a) for a in m) for m in mats]
    outs = [w4.w4_dequant_f16(*d, flags=w4.OVERLAP_PREVIOUS) for d in dev]
    torch.cuda.synchronize()
    for (N, K), (qw, s, b), o in zip(shapes, mats, outs):
        if N * K <= 4 * 1024 * 1024:
            assert np.array_equal(o.cpu().numpy().view(np.uint16), oracle.dequant_f16_t(qw, s, b, N, K))
        else:
            rows = np.array([0, 1, N // 3, N - 1], dtype=np.int32)
            want = oracle.dequant_f16_rows(qw, s, b, K, rows)
            assert np.array_equal(o.cpu().numpy().view(np.uint16)[:, rows].T, want)
