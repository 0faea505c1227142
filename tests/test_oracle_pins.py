"""Pins for the CPU oracle against facts that do not come from the oracle.

Each test checks an oracle function against something fixed by the pages'
definitions or by mathematics: hand-derived golden values (tests/golden/),
exhaustive comparison with numpy's binary16 conversions, exact rational
arithmetic (fractions.Fraction) on small cases, closed forms and invariants.
"""
import bisect
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import golden_lines


# ---------------------------------------------------------------- binary16

def _half_value(bits):
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


def test_half_decode_exhaustive():
    """All 65536 bit patterns decode exactly as numpy's float16 -> float64."""
    for h in range(1 << 16):
        ref = _half_value(h)
        got = oracle.half_to_double(h)
        if np.isnan(ref):
            assert np.isnan(got), hex(h)
        else:
            assert got == ref and np.signbit(got) == np.signbit(ref), hex(h)


def _encode_candidates():
    g = np.random.default_rng(7)
    finite = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (finite[:-1] + finite[1:]) / 2.0           # exact ties (binary64 has room)
    above = np.nextafter(mids, np.inf)
    below = np.nextafter(mids, -np.inf)
    rand = np.exp2(g.uniform(-27, 17, size=20000)) * g.choice([-1.0, 1.0], size=20000)
    edges = np.array([65504.0, 65519.999, 65520.0, 65536.0, 1e6, 2.0**-24, 2.0**-25,
                      3 * 2.0**-26, 2.0**-26, 0.0, -0.0, 2.0**-14, 2.0**-14 - 2.0**-25])
    v = np.concatenate([finite, mids, above, below, rand, edges])
    return np.concatenate([v, -v])


def test_half_encode_matches_numpy():
    """Correctly rounded binary64 -> binary16 (RNE) agrees bit for bit with numpy."""
    v = _encode_candidates()
    ref = v.astype(np.float16).view(np.uint16)
    got = oracle.double_to_half_array(v)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(v[i], hex(got[i]), hex(ref[i])) for i in bad[:5]]


_FINITE_POS = [Fraction(_half_value(h)) for h in range(0x7C00)]


def _rne_half_fraction(x: Fraction) -> int:
    """Round an exact rational to binary16 by brute force over the finite halves."""
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    top = Fraction(65520)  # max finite 65504 + half its spacing: ties go to 2^16 -> inf
    if a >= top:
        return sign | 0x7C00
    i = bisect.bisect_left(_FINITE_POS, a)
    if i < len(_FINITE_POS) and _FINITE_POS[i] == a:
        return sign | i
    lo, hi = i - 1, i
    dlo, dhi = a - _FINITE_POS[lo], _FINITE_POS[hi] - a
    if dlo < dhi or (dlo == dhi and lo % 2 == 0):
        return sign | lo
    return sign | hi


def test_half_encode_matches_fraction_rounding():
    g = np.random.default_rng(11)
    vals = np.exp2(g.uniform(-26, 16.5, size=3000)) * g.choice([-1.0, 1.0], size=3000)
    for v in vals:
        assert oracle.double_to_half(v) == _rne_half_fraction(Fraction(v)), v


# ---------------------------------------------------------------- unpack

def test_unpack_golden_nibble_order():
    for line in golden_lines("nibble_order.txt"):
        parts = line.split()
        word = int(parts[0], 16)
        want = [int(t) for t in parts[1:]]
        qw = np.array([[word]], dtype=np.uint32)
        got = oracle.unpack(qw, 1, 8)[0].tolist()
        assert got == want, (hex(word), got, want)


def test_unpack_matches_pack_roundtrip():
    g = np.random.default_rng(3)
    q = g.integers(0, 16, size=(5, 128), dtype=np.uint8)
    assert np.array_equal(oracle.unpack(synth.pack_nibbles(q), 5, 128), q)


# ---------------------------------------------------------------- dequant

def _one_group(word, s_bits, b_bits):
    qw = np.full((1, 8), word, dtype=np.uint32)
    s = np.array([[s_bits]], dtype=np.uint16)
    b = np.array([[b_bits]], dtype=np.uint16)
    return qw, s, b


def test_dequant_f16_golden():
    for line in golden_lines("dequant_f16.txt"):
        data = line.split(";")[0].split()
        s_bits, q, b_bits, want = int(data[0], 16), int(data[1]), int(data[2], 16), int(data[3], 16)
        qw, s, b = _one_group(q, s_bits, b_bits)   # code q at k=0, zeros elsewhere
        got = int(oracle.dequant_f16_rows(qw, s, b, 64, [0])[0, 0])
        assert got == want, (line, hex(got))


def _random_half_bits(g, n, lo_exp=0, hi_exp=30):
    e = g.integers(lo_exp, hi_exp + 1, size=n)
    f = g.integers(0, 1024, size=n)
    sgn = g.integers(0, 2, size=n)
    return ((sgn << 15) | (e << 10) | f).astype(np.uint16)


def test_dequant_exact_and_rounded_vs_fraction():
    """scale*q + bias exactly (binary64) and its binary16 rounding, for q = 0..15
    against a wide random spread of binary16 scales and biases (subnormals included)."""
    g = np.random.default_rng(5)
    N = 1024
    s = _random_half_bits(g, N)
    b = _random_half_bits(g, N)
    qw = np.zeros((N, 8), dtype=np.uint32)
    qw[:, 0] = 0x76543210
    qw[:, 1] = 0xFEDCBA98                       # k = 0..15 hold q = 0..15
    rows = np.arange(N)
    w = oracle.dequant_exact_rows(qw, s[:, None], b[:, None], 64, rows)
    w16 = oracle.dequant_f16_rows(qw, s[:, None], b[:, None], 64, rows)
    for n in range(N):
        sf = Fraction(_half_value(int(s[n])))
        bf = Fraction(_half_value(int(b[n])))
        for q in range(16):
            exact = sf * q + bf
            assert Fraction(w[n, q]) == exact
            if exact == 0:
                continue  # zero sign is pinned by the golden file
            assert int(w16[n, q]) == _rne_half_fraction(exact), (hex(s[n]), q, hex(b[n]))


def test_dequant_transposed_layout():
    qw, s, b = synth.make_linear(9, 24, 192)
    t = oracle.dequant_f16_t(qw, s, b, 24, 192)
    r = oracle.dequant_f16_rows(qw, s, b, 192, np.arange(24))
    assert t.shape == (192, 24)
    assert np.array_equal(t, r.T)


# ---------------------------------------------------------------- GEMV

def test_gemv_golden_worked_example():
    x = np.array([1.0] * 32 + [-0.5] * 32, dtype=np.float16)[None, :]
    lines = list(golden_lines("gemv_worked.txt"))
    qw = np.zeros((len(lines), 8), dtype=np.uint32)
    s = np.zeros((len(lines), 1), dtype=np.uint16)
    b = np.zeros((len(lines), 1), dtype=np.uint16)
    want_y, want_ad = [], []
    for line in lines:
        r, word, sb, bb, y, ad = line.split()
        r = int(r)
        qw[r, :] = int(word, 16)
        s[r, 0] = int(sb, 16)
        b[r, 0] = int(bb, 16)
        want_y.append(float(y))
        want_ad.append(float(ad))
    y, ad = oracle.gemv(x, qw, s, b, len(lines), 64)
    assert y[0].tolist() == want_y
    assert ad[0].tolist() == want_ad


def test_gemv_closed_form_q8_zero_bias():
    """All q = 8, bias = 0  =>  y[n] = 8 * sum_g scale[n][g] * sum_{k in g} x[k] (exact here)."""
    g = np.random.default_rng(21)
    N, K, M = 6, 512, 2
    qw = np.full((N, K // 8), 0x88888888, dtype=np.uint32)
    s, _ = synth.make_scales_biases(g, N, K)
    b = np.zeros_like(s)
    x = g.integers(-4, 5, size=(M, K)).astype(np.float16)
    y, _ = oracle.gemv(x, qw, s, b, N, K)
    for m in range(M):
        for n in range(N):
            want = sum(8 * Fraction(float(s[n, gi])) * sum(int(v) for v in x[m, gi * 64:(gi + 1) * 64])
                       for gi in range(K // 64))
            assert Fraction(y[m, n]) == want


@pytest.mark.parametrize("N,K,M", [(1, 64, 1), (3, 64, 2), (4, 128, 2), (2, 192, 1)])
def test_gemv_fraction_brute_force(N, K, M):
    """Tiny GEMVs against exact rational arithmetic from unpacked codes."""
    qw, s, b = synth.make_linear(100 + N * K + M, N, K)
    x = synth.make_x(200 + N, M, K)
    y, ad = oracle.gemv(x, qw, s, b, N, K)
    for n in range(N):
        for m in range(M):
            acc = Fraction(0)
            aacc = Fraction(0)
            for k in range(K):
                q = (int(qw[n, k // 8]) >> (4 * (k % 8))) & 0xF
                w = Fraction(float(s[n, k // 64])) * q + Fraction(float(b[n, k // 64]))
                p = w * Fraction(float(x[m, k]))
                acc += p
                aacc += abs(p)
            assert abs(Fraction(y[m, n]) - acc) <= Fraction(1, 10**12) * aacc
            assert abs(Fraction(ad[m, n]) - aacc) <= Fraction(1, 10**12) * aacc


def test_gemv_invariant_dequant_then_matmul():
    """Fused GEMV == (exact dequant) @ x computed with numpy's float64 matmul."""
    N, K, M = 37, 640, 3
    qw, s, b = synth.make_linear(31, N, K)
    x = synth.make_x(32, M, K)
    y, ad = oracle.gemv(x, qw, s, b, N, K)
    w = oracle.dequant_exact_rows(qw, s, b, K, np.arange(N))
    ref = x.astype(np.float64) @ w.T
    assert np.all(np.abs(y - ref) <= 1e-12 * ad)


def test_gemv_rows_subset_matches_full():
    N, K = 50, 256
    qw, s, b = synth.make_linear(41, N, K)
    x = synth.make_x(42, 2, K)
    y, _ = oracle.gemv(x, qw, s, b, N, K)
    rows = [49, 0, 17, 17]
    ys, _ = oracle.gemv_rows(x, qw, s, b, K, rows)
    assert np.array_equal(ys, y[:, rows])
    yt, _ = oracle.gemv(x, qw, s, b, N, K, threads=3)
    assert np.array_equal(yt, y)


# ---------------------------------------------------------------- top-k

def test_topk_golden():
    for line in golden_lines("topk_worked.txt"):
        lg, k, want = [p.split() for p in line.split(";")]
        idx, val = oracle.topk(np.array([float(t) for t in lg]), int(k[0]))
        assert idx.tolist() == [int(t) for t in want], line


def test_topk_brute_force_with_ties():
    g = np.random.default_rng(8)
    for trial in range(40):
        N = int(g.integers(1, 300))
        lg = g.integers(-20, 20, size=N).astype(np.float64) / 4.0   # many exact ties
        k = int(g.integers(1, min(N, 64) + 1))
        want = sorted(range(N), key=lambda i: (-lg[i], i))[:k]
        idx, val = oracle.topk(lg, k)
        assert idx.tolist() == want
        assert val.tolist() == [lg[i] for i in want]


def test_topk_k1_is_first_argmax_and_planted_max():
    g = np.random.default_rng(9)
    lg = g.standard_normal(151936)
    lg[12345] = 50.0
    lg[99999] = 50.0
    idx, val = oracle.topk(lg, 1)
    assert idx[0] == 12345 == int(np.argmax(lg))
    idx, _ = oracle.topk(lg, 3)
    assert idx[:2].tolist() == [12345, 99999]


# ---------------------------------------------------------------- GEMM

def test_gemm_closed_form_integers():
    """Integer-valued halves: the product is an exact integer matmul."""
    g = np.random.default_rng(12)
    M, N, K = 5, 7, 96
    x = g.integers(-8, 9, size=(M, K)).astype(np.float16)
    w = g.integers(-8, 9, size=(K, N)).astype(np.float16)
    y, ad = oracle.gemm(x, w, M, N, K)
    ref = x.astype(np.int64) @ w.astype(np.int64)
    assert np.array_equal(y, ref.astype(np.float64))
    assert np.array_equal(ad, np.abs(x.astype(np.int64)) @ np.abs(w.astype(np.int64)))
    ms, ns = [4, 0, 2], [6, 3, 0]
    ye, _ = oracle.gemm_entries(x, w, N, K, ms, ns)
    assert ye.tolist() == [y[m, n] for m, n in zip(ms, ns)]


def test_gemm_of_dequant_scratch_equals_gemv():
    """Dequant-once then dense GEMM equals the fused GEMV up to the binary16
    rounding of each weight (relative 2^-11 per term)."""
    N, K, M = 40, 320, 3
    qw, s, b = synth.make_linear(51, N, K)
    x = synth.make_x(52, M, K)
    yv, ad = oracle.gemv(x, qw, s, b, N, K)
    w16 = oracle.dequant_f16_t(qw, s, b, N, K)
    yg, adg = oracle.gemm(x, w16, M, N, K)
    assert np.all(np.abs(yg - yv) <= 2.0**-11 * ad + 1e-12)
    assert np.all(np.abs(adg - ad) <= 2.0**-11 * ad + 1e-12)


# ------------------------------------------------- group size and symmetric codes

def test_dequant_symmetric_vs_fraction():
    """Symmetric codes: scale*(q - 8) exactly (binary64) and its binary16
    rounding, q = 0..15, against a wide random spread of binary16 scales; an
    exact zero (q = 8) carries the sign of the IEEE product scale * (+0)."""
    g = np.random.default_rng(6)
    N = 1024
    s = _random_half_bits(g, N)
    qw = np.zeros((N, 8), dtype=np.uint32)
    qw[:, 0] = 0x76543210
    qw[:, 1] = 0xFEDCBA98                       # k = 0..15 hold q = 0..15
    rows = np.arange(N)
    w = oracle.dequant_exact_rows(qw, s[:, None], None, 64, rows)
    w16 = oracle.dequant_f16_rows(qw, s[:, None], None, 64, rows)
    for n in range(N):
        sf = Fraction(_half_value(int(s[n])))
        for q in range(16):
            exact = sf * (q - 8)
            assert Fraction(w[n, q]) == exact
            if exact == 0:
                assert int(w16[n, q]) == (int(s[n]) & 0x8000), hex(s[n])
            else:
                assert int(w16[n, q]) == _rne_half_fraction(exact), (hex(s[n]), q)
    # codes 16..63 (all zero words) are q = 0: w = -8 * scale
    assert np.array_equal(w[:, 16:], np.repeat(-8.0 * w[:, 9:10], 48, axis=1))


def test_dequant_symmetric_golden():
    for line in golden_lines("dequant_sym_f16.txt"):
        data = line.split(";")[0].split()
        s_bits, q, want = int(data[0], 16), int(data[1]), int(data[2], 16)
        qw = np.full((1, 8), q, dtype=np.uint32)   # code q at k = 0, zeros elsewhere
        s = np.array([[s_bits]], dtype=np.uint16)
        got = int(oracle.dequant_f16_rows(qw, s, None, 64, [0])[0, 0])
        assert got == want, (line, hex(got))


def _linear(seed, N, K, group, sym):
    if sym:
        return synth.make_linear_sym(seed, N, K, group)
    return synth.make_linear(seed, N, K, group)


@pytest.mark.parametrize("group,sym", [(32, False), (128, False), (256, False), (32, True), (64, True),
                                       (128, True), (256, True)])
def test_gemv_fraction_brute_force_formats(group, sym):
    """Tiny GEMVs of every supported format against exact rational arithmetic
    on the unpacked codes: the scale (and bias) of element k is entry k // group."""
    N, K, M = 3, 256, 2
    qw, s, b = _linear(300 + group + sym, N, K, group, sym)
    x = synth.make_x(400 + group, M, K)
    y, ad = oracle.gemv(x, qw, s, b, N, K, group=group)
    for n in range(N):
        for m in range(M):
            acc = Fraction(0)
            aacc = Fraction(0)
            for k in range(K):
                q = (int(qw[n, k // 8]) >> (4 * (k % 8))) & 0xF
                sc = Fraction(float(s[n, k // group]))
                w = sc * (q - 8) if sym else sc * q + Fraction(float(b[n, k // group]))
                p = w * Fraction(float(x[m, k]))
                acc += p
                aacc += abs(p)
            assert abs(Fraction(y[m, n]) - acc) <= Fraction(1, 10**12) * aacc
            assert abs(Fraction(ad[m, n]) - aacc) <= Fraction(1, 10**12) * aacc


@pytest.mark.parametrize("sym", [False, True])
def test_group_invariant_under_repeated_scales(sym):
    """A group-G weight equals the group-G/2 weight whose scales (and biases)
    are each repeated twice: the dequantised values bit for bit and the GEMV
    exactly, for G = 64 and 128."""
    N, K = 5, 512
    x = synth.make_x(51, 2, K)
    for G in (64, 128):
        qw, s, b = _linear(50 + G, N, K, G, sym)
        s2 = np.repeat(s, 2, axis=1)
        b2 = None if b is None else np.repeat(b, 2, axis=1)
        assert np.array_equal(oracle.dequant_f16_t(qw, s, b, N, K, group=G),
                              oracle.dequant_f16_t(qw, s2, b2, N, K, group=G // 2))
        y, _ = oracle.gemv(x, qw, s, b, N, K, group=G)
        y2, _ = oracle.gemv(x, qw, s2, b2, N, K, group=G // 2)
        assert np.array_equal(y, y2)


def test_symmetric_equals_affine_with_bias_minus_eight_scales():
    """Symmetric codes are the affine format with bias = -8 * scale (exact in
    binary16 for these scales): same dequantised bits, same GEMV."""
    N, K = 7, 384
    qw, s, _ = synth.make_linear_sym(61, N, K, 128)
    b = (-8.0 * s.astype(np.float64)).astype(np.float16)
    assert np.array_equal(b.astype(np.float64), -8.0 * s.astype(np.float64))
    assert np.array_equal(oracle.dequant_f16_t(qw, s, None, N, K, group=128),
                          oracle.dequant_f16_t(qw, s, b, N, K, group=128))
    x = synth.make_x(62, 3, K)
    y, _ = oracle.gemv(x, qw, s, None, N, K, group=128)
    ya, _ = oracle.gemv(x, qw, s, b, N, K, group=128)
    assert np.array_equal(y, ya)


def test_gemv_symmetric_closed_forms():
    """Symmetric codes: all q = 8 gives y = 0 exactly; all q = 9 gives
    y[n] = sum_g scale[n][g] * sum_{k in g} x[k] (exact for small integer x)."""
    g = np.random.default_rng(71)
    N, K, M, G = 4, 512, 2, 128
    s = g.uniform(0.002, 0.02, size=(N, K // G)).astype(np.float16)
    x = g.integers(-4, 5, size=(M, K)).astype(np.float16)
    q8 = np.full((N, K // 8), 0x88888888, dtype=np.uint32)
    y, _ = oracle.gemv(x, q8, s, None, N, K, group=G)
    assert np.all(y == 0.0)
    q9 = np.full((N, K // 8), 0x99999999, dtype=np.uint32)
    y, _ = oracle.gemv(x, q9, s, None, N, K, group=G)
    for m in range(M):
        for n in range(N):
            want = sum(Fraction(float(s[n, gi])) * sum(int(v) for v in x[m, gi * G:(gi + 1) * G])
                       for gi in range(K // G))
            assert Fraction(y[m, n]) == want
