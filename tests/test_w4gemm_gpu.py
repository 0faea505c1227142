"""w4_gemm (int4 GEMM with the dequantisation inside the tensor-core
pipeline, M <= 128) on the GPU against the CPU oracle.

Tolerance 1e-3 * sum_k |w_k x_k| + 1e-3 against the exact binary64 GEMV of
the oracle, for every activation row.  With a single K split the kernel
multiplies exactly the w4_dequant_f16 values in the f16_gemm operand layout,
so it is also compared bit for bit with that two-step path (a consistency
check between two GPU paths, beside the oracle parity)."""
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


def _linear(seed, N, K, group=64, sym=False):
    if sym:
        return synth.make_linear_sym(seed, N, K, group)
    return synth.make_linear(seed, N, K, group)


def _dv(a):
    return None if a is None else to_dev(a)


SMALL = [
    (1, 8, 64),         # one k step, one partial tile
    (5, 136, 128),      # ragged tile: 136 = 128 + 8
    (16, 256, 640),     # two whole tiles (sharing would save too few steps)
    (7, 1000, 2048),    # eight tiles, each shared by four blocks, ragged last tile
    (77, 1000, 896),
    (128, 2048, 2048),
    (128, 384, 11008),  # few tiles, long K: 22 blocks share each tile
    (64, 384, 11008),
    (5, 19584, 640),    # 153 tiles: one whole tile per block and a partial wave of one
    (33, 11008, 256),   # 86 whole tiles, nothing shared
]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_w4gemm_matches_oracle(w4, M, N, K):
    qw, s, b = _linear(8000 + N + K, N, K)
    x = synth.make_x(8100 + M, M, K)
    y = w4.w4_gemm(to_dev(x), to_dev(qw), to_dev(s), to_dev(b)).cpu().numpy()
    yo, ad = oracle.gemv(x, qw, s, b, N, K, threads=16)
    ok, worst = within_tol(y, yo, ad)
    assert ok, f"worst err/tol = {worst}"


@pytest.mark.parametrize("group,sym", [(32, False), (128, True), (256, False), (64, True), (32, True)])
def test_w4gemm_formats(w4, group, sym):
    M, N, K = 33, 512, 1024
    qw, s, b = _linear(8200 + group + sym, N, K, group, sym)
    x = synth.make_x(8201, M, K)
    y = w4.w4_gemm(to_dev(x), to_dev(qw), to_dev(s), _dv(b), group=group).cpu().numpy()
    yo, ad = oracle.gemv(x, qw, s, b, N, K, group=group, threads=16)
    ok, worst = within_tol(y, yo, ad)
    assert ok, f"worst err/tol = {worst}"


@pytest.mark.parametrize("M", [64, 128])
@pytest.mark.parametrize("group,sym", [(64, False), (128, True)])
def test_w4gemm_single_split_equals_dequant_then_gemm(w4, M, group, sym):
    """N = 22016 (172 tiles for 152 SMs: 152 whole tiles, the other 20 shared
    by blocks): the fused GEMM multiplies exactly the w4_dequant_f16 weight
    values, and only the order in which it adds its 64-k steps differs from
    f16_gemm on that scratch (a rotation per tile, partial sums of shared
    tiles), so every output is within one binary16 unit in the last place of
    f16_gemm's."""
    import torch
    N, K = 22016, 2048
    qw, s, b = _linear(8300 + M, N, K, group, sym)
    x = to_dev(synth.make_x(8301, M, K))
    args = (to_dev(qw), to_dev(s), _dv(b))
    y = w4.w4_gemm(x, *args, group=group)
    w16 = w4.w4_dequant_f16(*args, group=group)
    y2 = w4.f16_gemm(x, w16)
    ulps = (y.view(torch.int16).int() - y2.view(torch.int16).int()).abs()
    same_sign = (y.view(torch.int16) < 0) == (y2.view(torch.int16) < 0)
    close = (same_sign & (ulps <= 1)) | ((y.float() - y2.float()).abs() <= 1e-4)
    assert bool(close.all()), f"{int((~close).sum())} outputs differ by more than one unit in the last place"


FULL = sorted({(K, N) for _, K, N in synth.QWEN25_3B} | {(2048, 2560), (2048, 22016)})


@pytest.mark.parametrize("K,N", FULL)
@pytest.mark.parametrize("M", [16, 128])
def test_w4gemm_full_size_sampled(w4, M, K, N):
    qw, s, b = _linear(8400 + N + K, N, K)
    x = synth.make_x(8401 + M, M, K)
    y = w4.w4_gemm(to_dev(x), to_dev(qw), to_dev(s), to_dev(b)).cpu().numpy()
    g = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, 127, 128, N // 2, N - 1], g.integers(0, N, size=24)])).astype(np.int32)
    yo, ad = oracle.gemv_rows(x, qw, s, b, K, rows)
    ok, worst = within_tol(y[:, rows], yo, ad)
    assert ok, f"worst err/tol = {worst}"


@pytest.mark.parametrize("M", [16, 64])
def test_w4gemm_repeated_calls_share_a_workspace(w4, M):
    """Shared tiles (summed by the last sharer at M = 16, in slices after the
    sharers' flags at M = 64): counters and flags are left ready after every
    call, so one zero-filled workspace serves many calls with identical
    results."""
    import torch
    N, K = 1024, 4096
    qw, s, b = _linear(8500, N, K)
    x = synth.make_x(8501, M, K)
    ws = w4.w4_gemm_workspace(M, N, K)
    args = (to_dev(x), to_dev(qw), to_dev(s), to_dev(b))
    ys = [w4.w4_gemm(*args, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
    yo, ad = oracle.gemv(x, qw, s, b, N, K, threads=16)
    ok, worst = within_tol(ys[0].cpu().numpy(), yo, ad)
    assert ok, f"worst err/tol = {worst}"


def test_w4gemm_both_sharing_forms_alternate_on_one_workspace(w4):
    """Calls at M = 64 (flags) and M = 16 (arrival counters) alternate on one
    workspace, back to back on a stream: each form leaves its own counters
    ready for the next call of either form."""
    import torch
    N, K = 2048, 2048
    qw, s, b = _linear(8550, N, K)
    xs = {M: synth.make_x(8551 + M, M, K) for M in (16, 64)}
    ws = w4.w4_gemm_workspace(64, N, K)
    args = (to_dev(qw), to_dev(s), to_dev(b))
    outs = {16: [], 64: []}
    for _ in range(3):
        for M in (64, 16):
            outs[M].append(w4.w4_gemm(to_dev(xs[M]), *args, workspace=ws))
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    for M in (16, 64):
        assert all(torch.equal(outs[M][0], o) for o in outs[M][1:])
        yo, ad = oracle.gemv(xs[M], qw, s, b, N, K, threads=16)
        ok, worst = within_tol(outs[M][0].cpu().numpy(), yo, ad)
        assert ok, f"M={M}: worst err/tol = {worst}"


def test_w4gemm_overlap_flag_keeps_the_activation_dependency(w4):
    """With OVERLAP_PREVIOUS the weight tiles are fetched and converted early,
    but x written by the previous kernel on the stream is read after it."""
    import torch
    M, N, K = 32, 2560, 2048
    qw, s, b = _linear(8600, N, K)
    x_new = synth.make_x(8601, M, K)
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    ws = w4.w4_gemm_workspace(M, N, K)
    src = to_dev(x_new)
    args = (to_dev(qw), to_dev(s), to_dev(b))
    torch.cuda.synchronize()
    for _ in range(3):
        x.zero_()
        x.copy_(src)  # the previous kernel writes x
        y = w4.w4_gemm(x, *args, workspace=ws, flags=w4.OVERLAP_PREVIOUS)
    torch.cuda.synchronize()
    yo, ad = oracle.gemv(x_new, qw, s, b, N, K, threads=16)
    ok, worst = within_tol(y.cpu().numpy(), yo, ad)
    assert ok, f"worst err/tol = {worst}"
