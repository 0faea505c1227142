"""lm_head_argmax_topk on the GPU against the CPU oracle's full logits.

Indices must match exactly wherever the oracle ranking separates neighbours
by more than their float tolerances; the other positions are excluded,
counted, and checked for validity."""
import numpy as np
import pytest

import oracle
import synth
from _gpu import require_gpu, to_dev, topk_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    require_gpu()
    import int4_weight_only_affine_gb300 as w4
    return w4


def _run(w4, seed, M, N, K, k, rows_full=None):
    import torch
    qw, s, b = synth.make_linear(seed, N, K)
    x = synth.make_x(seed + 1, M, K)
    ws = torch.randint(0, 255, (w4.lm_head_workspace_bytes(M, N, k),), dtype=torch.uint8, device="cuda")
    idx, val = w4.lm_head_argmax_topk(to_dev(x), to_dev(qw), to_dev(s), to_dev(b), k=k, workspace=ws)
    idx, val = idx.cpu().numpy(), val.cpu().numpy()
    check_rows = range(M) if rows_full is None else rows_full
    excluded = 0
    for m in check_rows:
        lg, ad = oracle.gemv(x[m:m + 1], qw, s, b, N, K, threads=16)
        excluded += topk_check(idx[m], val[m], lg[0], ad[0], k)
    # Rows not checked in full: returned values equal the oracle logit of the returned index.
    for m in set(range(M)) - set(check_rows):
        lg, ad = oracle.gemv_rows(x[m:m + 1], qw, s, b, K, idx[m])
        assert np.all(np.abs(val[m] - lg[0]) <= 1e-3 * ad[0] + 1e-3)
    return idx, val, excluded


@pytest.mark.parametrize("M,N,K,k", [
    (1, 1000, 896, 1), (1, 1000, 896, 5),      # single-GEMV case with top-5
    (3, 257, 192, 1), (3, 257, 192, 7), (2, 257, 192, 64),
    (16, 17, 64, 16), (9, 130, 128, 3), (16, 4096, 256, 1), (5, 3000, 512, 33),
])
def test_topk_small(w4, M, N, K, k):
    _run(w4, 40 + N + k, M, N, K, k)


def test_topk_ties_lowest_index(w4):
    """Rows with identical weights give identical logits: ties go to the lowest index."""
    import torch
    N, K = 600, 128
    qw, s, b = synth.make_linear(5, N, K)
    x = synth.make_x(6, 1, K)
    # Rows 7, 100, 333, 599 get the same codes, maximising x . w: equal logits.
    code = np.where(x[0].astype(np.float64) > 0, 15, 0).astype(np.uint8)
    row = synth.pack_nibbles(code[None, :])[0]
    ones = np.full(K // 64, 0x3C00, dtype=np.uint16).view(np.float16)
    for r in (7, 100, 333, 599):
        qw[r] = row
        s[r] = ones
        b[r] = np.zeros(K // 64, dtype=np.float16)
    idx, val = w4.lm_head_argmax_topk(to_dev(x), to_dev(qw), to_dev(s), to_dev(b), k=4)
    assert idx.cpu().numpy()[0].tolist() == [7, 100, 333, 599]
    assert len(set(val.cpu().numpy()[0].tolist())) == 1


@pytest.mark.parametrize("K,k", [(1024, 1), (2048, 1), (2048, 50)])
def test_topk_full_vocab(w4, K, k):
    _run(w4, 500 + K + k, 1, 151936, K, k)


@pytest.mark.parametrize("M", [2, 4, 8, 16])
def test_argmax_full_vocab_batched(w4, M):
    """Per-row greedy argmax at the 3B head shape; two rows checked against the
    full oracle logits, the rest on the returned entries."""
    _run(w4, 900 + M, M, 151936, 2048, 1, rows_full=[0, M - 1])


def test_topk_deterministic(w4):
    import torch
    N, K, M, k = 151936, 2048, 1, 50
    qw, s, b = synth.make_linear(3, N, K)
    x = synth.make_x(4, M, K)
    a = [to_dev(x), to_dev(qw), to_dev(s), to_dev(b)]
    i1, v1 = w4.lm_head_argmax_topk(*a, k=k)
    i2, v2 = w4.lm_head_argmax_topk(*a, k=k)
    assert torch.equal(i1, i2) and torch.equal(v1, v2)
