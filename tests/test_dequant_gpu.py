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


@pytest.mark.parametrize("N,K", [(1000, 896), (257, 192), (1, 64), (64, 64), (130, 128), (8, 640), (3, 1024)])
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
