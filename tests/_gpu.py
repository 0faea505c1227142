"""Helpers shared by the GPU parity tests (not collected: no test_ prefix)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

TOL_REL = 1e-3
TOL_ABS = 1e-3

# (test id, excluded positions, checked positions) of every top-k comparison
# in this session; printed in the terminal summary (tests/conftest.py).
EXCLUSIONS = []


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def dev():
    return torch.device("cuda:0")


def to_dev(a: np.ndarray):
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def within_tol(got, want, absdot):
    """|gpu - oracle| <= 1e-3 * sum_k |w_k x_k| + 1e-3 elementwise; returns (ok, worst ratio)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    tol = TOL_REL * absdot + TOL_ABS
    return bool(np.all(err <= tol)), float(np.max(err / tol)) if err.size else 0.0


def undecidable_positions(logits, absdot, k):
    """Rank positions 0..k-1 of the oracle ranking that the float tolerance
    cannot decide: a neighbour (in the oracle top k+1) lies within the sum of
    the two logits' tolerances.  Depends on the oracle only."""
    import oracle
    oi, ov = oracle.topk(logits, min(k + 1, logits.size))
    tol = TOL_REL * absdot + TOL_ABS
    out = []
    for p in range(k):
        near_prev = p > 0 and ov[p - 1] - ov[p] <= tol[oi[p - 1]] + tol[oi[p]]
        near_next = p + 1 < len(oi) and ov[p] - ov[p + 1] <= tol[oi[p]] + tol[oi[p + 1]]
        if near_prev or near_next:
            out.append(p)
    return out, oi, ov


def topk_check(gpu_idx, gpu_val, logits, absdot, k):
    """Compare a GPU top-k with oracle logits of one row.

    Positions whose oracle neighbours (in the oracle ranking) are separated by
    more than the sum of their tolerances must match index for index; the
    other positions are counted as excluded and must still be valid: the GPU's
    index there has an oracle logit within tolerance of the oracle's value at
    that rank.  Returned values must be within tolerance of the oracle logit
    of the returned index.  Returns the number of excluded positions."""
    excl, oi, ov = undecidable_positions(logits, absdot, k)
    tol = TOL_REL * absdot + TOL_ABS
    for p in range(k):
        i_gpu = int(gpu_idx[p])
        assert 0 <= i_gpu < logits.size
        assert abs(float(gpu_val[p]) - logits[i_gpu]) <= tol[i_gpu], (p, i_gpu)
        if p not in excl:
            assert i_gpu == int(oi[p]), (p, i_gpu, int(oi[p]))
        else:
            assert abs(logits[i_gpu] - ov[p]) <= tol[i_gpu] + tol[oi[p]], (p, i_gpu)
    assert len(set(int(i) for i in gpu_idx[:k])) == k, "duplicate indices"
    return len(excl)


def note_exclusions(request, excluded, positions):
    """Record a test's excluded / checked top-k positions (junit properties and
    the terminal summary)."""
    request.node.user_properties.append(("topk_excluded", excluded))
    request.node.user_properties.append(("topk_positions", positions))
    EXCLUSIONS.append((request.node.nodeid, excluded, positions))


def plant_topk(qw, s, b, x_row, rows, scales, group, sym):
    """Plants rows whose logits under activation row x_row are far above any
    other and strictly ordered: row rows[i] gets code 15 where x_row > 0 and 0
    elsewhere, scale scales[i] in every group and bias 0, so its logit is
    scales[i] * 15 * sum_{x>0} x (affine) or scales[i] * (7 * sum_{x>0} x +
    8 * sum_{x<0} |x|) (symmetric), every product w*x >= 0.  Modifies the
    arrays in place."""
    import synth
    K = x_row.size
    code = np.where(x_row.astype(np.float64) > 0, 15, 0).astype(np.uint8)
    packed = synth.pack_nibbles(code[None, :])[0]
    for r, sc in zip(rows, scales):
        qw[r] = packed
        s[r] = np.float16(sc)
        if not sym:
            b[r] = np.float16(0.0)
