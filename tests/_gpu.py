"""Helpers shared by the GPU parity tests (not collected: no test_ prefix)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

TOL_REL = 1e-3
TOL_ABS = 1e-3


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


def topk_check(gpu_idx, gpu_val, logits, absdot, k):
    """Compare a GPU top-k with oracle logits of one row.

    Positions whose oracle neighbours (in the oracle ranking) are separated by
    more than the sum of their tolerances must match index for index; the
    other positions are counted as excluded and must still be valid: the GPU's
    index there has an oracle logit within tolerance of the oracle's value at
    that rank.  Returned values must be within tolerance of the oracle logit
    of the returned index.  Returns the number of excluded positions."""
    import oracle
    oi, ov = oracle.topk(logits, min(k + 1, logits.size))
    tol = TOL_REL * absdot + TOL_ABS
    excluded = 0
    for p in range(k):
        i_gpu = int(gpu_idx[p])
        assert 0 <= i_gpu < logits.size
        assert abs(float(gpu_val[p]) - logits[i_gpu]) <= tol[i_gpu], (p, i_gpu)
        decidable = True
        if p > 0 and ov[p - 1] - ov[p] <= tol[oi[p - 1]] + tol[oi[p]]:
            decidable = False
        if p + 1 < len(oi) and ov[p] - ov[p + 1] <= tol[oi[p]] + tol[oi[p + 1]]:
            decidable = False
        if decidable:
            assert i_gpu == int(oi[p]), (p, i_gpu, int(oi[p]))
        else:
            excluded += 1
            assert abs(logits[i_gpu] - ov[p]) <= tol[i_gpu] + tol[oi[p]], (p, i_gpu)
    assert len(set(int(i) for i in gpu_idx[:k])) == k, "duplicate indices"
    return excluded
