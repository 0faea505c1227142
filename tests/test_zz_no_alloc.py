"""The no-allocation lm_head entry point (lm_head_argmax_topk_noalloc).

Some callers cannot allocate device memory where they run token selection:
allocator or memory-pool callbacks, processes held to a fixed memory budget,
embeddings that bring no allocator.  For them the library offers a variant of
lm_head_argmax_topk whose candidate buffer is a fixed array inside the
library.  These tests call it through the C ABI, two calls in a row, and
compare each result with the workspace-taking entry point; one sequence runs
a large selection and then a small one, so the small call meets the large
call's leftovers in the shared array.  The file is named to run after every
other test; it also passes in a fresh process (its first call performs the
per-device set-up)."""
import ctypes

import numpy as np
import pytest

import synth
from _gpu import require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    require_gpu()
    import int4_weight_only_affine_gb300 as w4
    P, I = ctypes.c_void_p, ctypes.c_int
    w4.lib.lm_head_argmax_topk_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P]
    w4.lib.lm_head_argmax_topk_noalloc.restype = I
    return w4


def _case(M, N, K, k):
    qw, s, b = synth.make_linear(700 + k + N % 97, N, K)
    x = synth.make_x(701 + M, M, K)
    return [to_dev(a) for a in (x, qw, s, b)]


def _noalloc(w4, args, M, N, K, k):
    import torch
    tx, tq, ts, tb = args
    idx = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    val = torch.full((M, k), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = w4.lib.lm_head_argmax_topk_noalloc(tx.data_ptr(), tq.data_ptr(), ts.data_ptr(), tb.data_ptr(),
                                            M, N, K, 64, k, idx.data_ptr(), val.data_ptr(), stream)
    assert st == 0, w4.lib.w4a16_status_string(st)
    torch.cuda.synchronize()
    return idx, val


def _same(w4, args, M, N, K, k, idx, val):
    import torch
    ref_idx, ref_val = w4.lm_head_argmax_topk(*args, k=k)
    assert torch.equal(idx, ref_idx)
    got, want = val.cpu().numpy().astype(np.float64), ref_val.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-3 * np.abs(want) + 1e-3)


@pytest.mark.parametrize("M,N,K,k", [(1, 151936, 2048, 50), (16, 151936, 2048, 1), (3, 1000, 896, 5)])
def test_noalloc_matches_workspace_entry_point(w4, M, N, K, k):
    args = _case(M, N, K, k)
    for _ in range(2):   # the shared array keeps the previous call's contents
        idx, val = _noalloc(w4, args, M, N, K, k)
        _same(w4, args, M, N, K, k, idx, val)


def test_noalloc_small_after_large(w4):
    """A large selection fills most of the shared array, then a small one runs
    on top of its leftovers (nothing in the array needs to start at zero)."""
    big, small = (16, 151936, 2048, 64), (3, 1000, 896, 5)
    a_big, a_small = _case(*big), _case(*small)
    idx, val = _noalloc(w4, a_big, *big)
    _same(w4, a_big, *big, idx, val)
    idx, val = _noalloc(w4, a_small, *small)
    _same(w4, a_small, *small, idx, val)


def test_noalloc_rejects_bad_sizes(w4):
    f = 0x10000
    lib = w4.lib
    assert lib.lm_head_argmax_topk_noalloc(f, f, f, f, 17, 1000, 64, 64, 1, f, f, None) == 2   # M > 16
    assert lib.lm_head_argmax_topk_noalloc(f, f, f, f, 1, 1000, 64, 64, 65, f, f, None) == 2   # k > 64
