"""lm_head_argmax_topk on the GPU against the CPU oracle's full logits.

Indices must match exactly wherever the oracle ranking separates neighbours
by more than their float tolerances; the other positions are excluded,
counted (printed in the terminal summary), bounded per case, and checked for
validity.  Random logits crowd the top of the ranking, so at large k most
positions are near-ties; the planted cases below give every one of the k
ranks a margin of several tolerances, so the whole index order is checked
exactly, at the full 151,936-row vocabulary, for M = 1 and M = 16, in the
affine group-64 and the symmetric group-128 formats, and with exact ties
inside the top 50 (ties go to the lowest index)."""
import numpy as np
import pytest

import oracle
import synth
from _gpu import note_exclusions, plant_topk, require_gpu, to_dev, topk_check, undecidable_positions

pytestmark = pytest.mark.gpu

VOCAB, HEAD_K = 151936, 2048


@pytest.fixture(scope="module")
def w4():
    require_gpu()
    import int4_weight_only_affine_gb300 as w4
    return w4


def _select(w4, x, qw, s, b, k, group=64):
    import torch
    M, K = x.shape
    N = qw.shape[0]
    ws = torch.randint(0, 255, (w4.lm_head_workspace_bytes(M, N, k),), dtype=torch.uint8, device="cuda")
    idx, val = w4.lm_head_argmax_topk(to_dev(x), to_dev(qw), to_dev(s), None if b is None else to_dev(b), k=k,
                                      workspace=ws, group=group)
    return idx.cpu().numpy(), val.cpu().numpy()


def _run(w4, seed, M, N, K, k, rows_full=None):
    qw, s, b = synth.make_linear(seed, N, K)
    x = synth.make_x(seed + 1, M, K)
    idx, val = _select(w4, x, qw, s, b, k)
    check_rows = range(M) if rows_full is None else rows_full
    excluded = 0
    for m in check_rows:
        lg, ad = oracle.gemv(x[m:m + 1], qw, s, b, N, K, threads=16)
        excluded += topk_check(idx[m], val[m], lg[0], ad[0], k)
    # Rows not checked in full: returned values equal the oracle logit of the returned index.
    for m in set(range(M)) - set(check_rows):
        lg, ad = oracle.gemv_rows(x[m:m + 1], qw, s, b, K, idx[m])
        assert np.all(np.abs(val[m] - lg[0]) <= 1e-3 * ad[0] + 1e-3)
    return idx, val, excluded, len(check_rows) * k


# max_excl: the oracle's own count of near-tie positions for these seeded
# inputs (it does not depend on the GPU); a larger count means the inputs
# changed.
@pytest.mark.parametrize("M,N,K,k,max_excl", [
    (1, 1000, 896, 1, 0), (1, 1000, 896, 5, 4),      # single-GEMV case with top-5
    (3, 257, 192, 1, 0), (3, 257, 192, 7, 1), (2, 257, 192, 64, 98),
    (16, 17, 64, 16, 40), (9, 130, 128, 3, 2), (16, 4096, 256, 1, 1), (5, 3000, 512, 33, 138),
])
def test_topk_small(w4, request, M, N, K, k, max_excl):
    _, _, excluded, positions = _run(w4, 40 + N + k, M, N, K, k)
    note_exclusions(request, excluded, positions)
    assert excluded <= max_excl


def test_topk_ties_lowest_index(w4):
    """Rows with identical weights give identical logits: ties go to the lowest index."""
    N, K = 600, 128
    qw, s, b = synth.make_linear(5, N, K)
    x = synth.make_x(6, 1, K)
    # Rows 7, 100, 333, 599 get the same codes, maximising x . w: equal logits.
    rows = (7, 100, 333, 599)
    plant_topk(qw, s, b, x[0], rows, [1.0] * 4, 64, False)
    idx, val = _select(w4, x, qw, s, b, 4)
    assert idx[0].tolist() == list(rows)
    assert len(set(val[0].tolist())) == 1


@pytest.mark.parametrize("K,k,max_excl", [(1024, 1, 0), (2048, 1, 0), (2048, 50, 49)])
def test_topk_full_vocab(w4, request, K, k, max_excl):
    _, _, excluded, positions = _run(w4, 500 + K + k, 1, VOCAB, K, k)
    note_exclusions(request, excluded, positions)
    assert excluded <= max_excl


# Oracle near-ties at the argmax of the two checked rows (0 and M - 1).
@pytest.mark.parametrize("M,max_excl", [(2, 2), (4, 0), (8, 1), (16, 0)])
def test_argmax_full_vocab_batched(w4, request, M, max_excl):
    """Per-row greedy argmax at the 3B head shape; two rows checked against the
    full oracle logits, the rest on the returned entries."""
    _, _, excluded, positions = _run(w4, 900 + M, M, VOCAB, HEAD_K, 1, rows_full=[0, M - 1])
    note_exclusions(request, excluded, positions)
    assert excluded <= max_excl


# ------------------------------------------------------------------ planted rankings

def _graded(k):
    """k scales 1, 0.99, ..., each rank's logit >= 1 % above the next: with
    every product w*x >= 0 the tolerance of a planted logit L is 1e-3*L +
    1e-3, so neighbours differ by at least 3x the sum of their tolerances."""
    return [1.0 - 0.01 * i for i in range(k)]


def _planted_case(seed, M, N, K, k, group, sym):
    """Seeded weights and activations with k planted rows per activation row
    (distinct rows for every activation row; see plant_topk)."""
    if sym:
        qw, s, b = synth.make_linear_sym(seed, N, K, group)
    else:
        qw, s, b = synth.make_linear(seed, N, K, group)
    x = synth.make_x(seed + 1, M, K)
    picks = np.random.default_rng(seed + 2).choice(N, size=M * k, replace=False).reshape(M, k)
    for m in range(M):
        plant_topk(qw, s, b, x[m], picks[m], _graded(k), group, sym)
    return qw, s, b, x, picks


def _check_all_decidable(w4, request, seed, M, N, K, k, group, sym):
    qw, s, b, x, picks = _planted_case(seed, M, N, K, k, group, sym)
    idx, val = _select(w4, x, qw, s, b, k, group)
    lg, ad = oracle.gemv(x, qw, s, b, N, K, group=group, threads=16)
    excluded = 0
    for m in range(M):
        und, oi, _ = undecidable_positions(lg[m], ad[m], k)
        assert und == [], f"row {m}: planted ranking has near-ties at {und}"
        # The oracle's ranking is the planted order.
        assert oi[:k].tolist() == picks[m].tolist()
        excluded += topk_check(idx[m], val[m], lg[m], ad[m], k)
        assert idx[m].tolist() == picks[m].tolist()
    note_exclusions(request, excluded, M * k)
    assert excluded == 0


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("group,sym", [(64, False), (128, True)])
def test_topk50_full_vocab_planted(w4, request, M, group, sym):
    """Top-50 over the 151,936-row head with all 50 ranks decidable: the GPU
    index order must equal the oracle's at every position of every row."""
    _check_all_decidable(w4, request, 8100 + M + group, M, VOCAB, HEAD_K, 50, group, sym)


@pytest.mark.parametrize("M", [2, 4, 8, 16])
def test_argmax_full_vocab_batched_planted(w4, request, M):
    """Per-row greedy argmax at the 3B head shape with a decidable winner in
    every activation row (all rows checked against the full oracle)."""
    _check_all_decidable(w4, request, 8200 + M, M, VOCAB, HEAD_K, 1, 64, False)


def test_topk5_single_gemv_planted(w4, request):
    """The 1000-row, K = 896 selection case with all 5 ranks decidable."""
    _check_all_decidable(w4, request, 8300, 1, 1000, 896, 5, 64, False)


def test_topk50_full_vocab_exact_ties(w4, request):
    """Ten groups of five identical rows fill the top 50: inside a group the
    logits tie exactly (on the GPU and in the oracle), between groups the
    margin is decidable.  The order must be group by group, lowest index
    first inside each group, exactly as the oracle ranks it."""
    N, K, k = VOCAB, HEAD_K, 50
    qw, s, b = synth.make_linear(8400, N, K)
    x = synth.make_x(8401, 1, K)
    picks = np.random.default_rng(8402).choice(N, size=k, replace=False)
    scales = [1.0 - 0.05 * (i // 5) for i in range(k)]
    plant_topk(qw, s, b, x[0], picks, scales, 64, False)
    idx, val = _select(w4, x, qw, s, b, k)
    lg, ad = oracle.gemv(x, qw, s, b, N, K, threads=16)
    oi, ov = oracle.topk(lg[0], k + 1)
    tol = 1e-3 * ad[0] + 1e-3
    expect = []
    for g in range(10):
        grp = sorted(int(r) for r in picks[5 * g:5 * g + 5])
        assert len({lg[0][r] for r in grp}) == 1, "planted rows must tie exactly in the oracle"
        expect += grp
    for p in range(k):   # decidable between groups (and from the rest of the vocabulary)
        if p % 5 == 4:
            assert ov[p] - ov[p + 1] > tol[oi[p]] + tol[oi[p + 1]]
    assert oi.tolist()[:k] == expect
    assert idx[0].tolist() == expect
    for g in range(10):
        assert len(set(val[0][5 * g:5 * g + 5].tolist())) == 1, "tied rows must give identical values"
    assert np.all(np.abs(val[0] - lg[0][idx[0]]) <= tol[idx[0]])
    note_exclusions(request, 0, k)


def test_topk_deterministic(w4):
    import torch
    N, K, M, k = VOCAB, HEAD_K, 1, 50
    qw, s, b = synth.make_linear(3, N, K)
    x = synth.make_x(4, M, K)
    a = [to_dev(x), to_dev(qw), to_dev(s), to_dev(b)]
    i1, v1 = w4.lm_head_argmax_topk(*a, k=k)
    i2, v2 = w4.lm_head_argmax_topk(*a, k=k)
    assert torch.equal(i1, i2) and torch.equal(v1, v2)
