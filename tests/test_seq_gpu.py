"""w4_gemv_seq (a list of GEMVs in one persistent launch) against the oracle.

Chained operations read the previous operation's output: the oracle runs the
same chain in binary64 and rounds each intermediate to binary16 itself, so no
GPU result is ever an oracle input."""
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


def _oracle_chain(M, x0, mats, chain):
    """Oracle outputs (binary64) and absdots of each op; chained ops take the
    previous op's output rounded to binary16 as x."""
    outs, ads, xs = [], [], []
    x = x0
    for i, ((qw, s, b, N, K), ch) in enumerate(zip(mats, chain)):
        if ch:
            x = oracle.double_to_half_array(outs[-1].ravel()).reshape(M, -1).view(np.float16)
        elif i > 0:
            x = synth.make_x(900 + i, M, K)
        y, ad = oracle.gemv(x, qw, s, b, N, K, threads=16)
        xs.append(x)
        outs.append(y)
        ads.append(ad)
    return outs, ads, xs


@pytest.mark.parametrize("M", [1, 4, 16])
def test_seq_chain_matches_oracle(w4, M):
    import torch
    # (K, N, chained to previous)
    plan = [(2048, 2560, False), (2560, 2048, True), (2048, 1024, True), (1024, 512, True), (512, 768, False),
            (768, 256, True)]
    mats = [synth.make_linear(1200 + i, N, K) + (N, K) for i, (K, N, _) in enumerate(plan)]
    chain = [c for _, _, c in plan]
    x0 = synth.make_x(77, M, plan[0][0])
    outs, ads, xs = _oracle_chain(M, x0, mats, chain)
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _, N, _ in plan]
    ops = []
    for i, ((qw, s, b, N, K), c) in enumerate(zip(mats, chain)):
        x = ys[i - 1] if c else to_dev(xs[i])
        ops.append((x, to_dev(qw), to_dev(s), to_dev(b), ys[i], c))
    w4.w4_gemv_seq(ops)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    for i in range(len(plan)):
        ok, worst = within_tol(ys[i].cpu().numpy(), outs[i], ads[i])
        assert ok, f"op {i}: worst err/tol = {worst}"


@pytest.mark.parametrize("M", [1, 3])
def test_seq_single_tiles_split_by_k(w4, M):
    """Operations with at most one 16-row tile per CTA and several 2048-k
    chunks, where a CTA's two warp teams take alternate chunks of its tile:
    K = 6144 (three chunks: the teams get two and one), chained to the
    previous output through the tagged exchange, with a ragged last tile
    (N = 2040), and K = 4096 after it; every output against the oracle."""
    import torch
    plan = [(2048, 6144, False), (6144, 2040, True), (4096, 2048, False)]
    mats = [synth.make_linear(1300 + i, N, K) + (N, K) for i, (K, N, _) in enumerate(plan)]
    chain = [c for _, _, c in plan]
    x0 = synth.make_x(78, M, plan[0][0])
    outs, ads, xs = _oracle_chain(M, x0, mats, chain)
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _, N, _ in plan]
    ops = []
    for i, ((qw, s, b, N, K), c) in enumerate(zip(mats, chain)):
        x = ys[i - 1] if c else to_dev(xs[i])
        ops.append((x, to_dev(qw), to_dev(s), to_dev(b), ys[i], c))
    w4.w4_gemv_seq(ops)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    for i in range(len(plan)):
        ok, worst = within_tol(ys[i].cpu().numpy(), outs[i], ads[i])
        assert ok, f"op {i}: worst err/tol = {worst}"


@pytest.mark.parametrize("mode", ["tagged", "counter"])
def test_seq_chain_repeated_calls_share_a_workspace(w4, mode):
    """Three calls on one workspace: the tagged exchange (words carry an
    (epoch, operation) tag) and the completion-counter fallback (a 16-byte
    workspace) give the oracle's results every time, so each launch resets
    the counters and a word left by the previous launch is never taken."""
    import torch
    M = 2
    plan = [(1024, 2048, False), (2048, 1024, True), (1024, 1536, True), (1536, 512, True)]
    mats = [synth.make_linear(1300 + i, N, K) + (N, K) for i, (K, N, _) in enumerate(plan)]
    chain = [c for _, _, c in plan]
    outs, ads, xs = _oracle_chain(M, synth.make_x(78, M, plan[0][0]), mats, chain)
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _, N, _ in plan]
    ops = [((ys[i - 1] if c else to_dev(xs[i])), to_dev(qw), to_dev(s), to_dev(b), ys[i], c)
           for i, ((qw, s, b, N, K), c) in enumerate(zip(mats, chain))]
    if mode == "tagged":
        ws = w4.seq_workspace(ops)
        assert ws.numel() == 16 + 4 * M * (2048 + 1024 + 1536)
    else:
        ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    for call in range(3):
        for y in ys:
            y.fill_(float("nan"))
        w4.w4_gemv_seq(ops, workspace=ws)
        torch.cuda.synchronize()
        assert w4.device_status() == 0
        for i in range(len(plan)):
            ok, worst = within_tol(ys[i].cpu().numpy(), outs[i], ads[i])
            assert ok, f"call {call} op {i}: worst err/tol = {worst}"
    head = ws[:12].cpu().numpy().view(np.uint32)
    assert head[0] == 0 and head[2] == 0 and head[1] == 3  # counters reset, epoch advanced once per launch


def test_seq_reads_a_prefix_of_the_previous_output(w4):
    """M = 1: an operation whose x is the first K elements of the previous
    output (K < N), as a projection reading part of a fused q|k|v output."""
    import torch
    M = 1
    plan = [(2048, 2560), (2048, 1024), (512, 768)]
    mats = [synth.make_linear(1400 + i, N, K) + (N, K) for i, (K, N) in enumerate(plan)]
    x0 = synth.make_x(79, M, 2048)
    y0, ad0 = oracle.gemv(x0, *mats[0][:3], 2560, 2048, threads=16)
    x1 = oracle.double_to_half_array(y0.ravel()[:2048]).reshape(1, 2048).view(np.float16)
    y1, ad1 = oracle.gemv(x1, *mats[1][:3], 1024, 2048, threads=16)
    x2 = oracle.double_to_half_array(y1.ravel()[:512]).reshape(1, 512).view(np.float16)
    y2, ad2 = oracle.gemv(x2, *mats[2][:3], 768, 512, threads=16)
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _, N in plan]
    ops = [(to_dev(x0), *[to_dev(a) for a in mats[0][:3]], ys[0], False),
           (ys[0][:, :2048], *[to_dev(a) for a in mats[1][:3]], ys[1], True),
           (ys[1][:, :512], *[to_dev(a) for a in mats[2][:3]], ys[2], True)]
    ws = w4.seq_workspace(ops)
    assert ws.numel() == 16 + 4 * (2560 + 1024)
    w4.w4_gemv_seq(ops, workspace=ws)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    for y, yo, ad in ((ys[0], y0, ad0), (ys[1], y1, ad1), (ys[2], y2, ad2)):
        ok, worst = within_tol(y.cpu().numpy(), yo, ad)
        assert ok, worst


def test_seq_long_list_crosses_launches(w4):
    """More operations than one launch carries (96): every even op reads the
    previous op's output, including op 96, whose producer ran in the previous
    launch.  Chains stay two long so values stay in binary16 range (a long
    chain of these synthetic weights grows by about 1.4x per step)."""
    import torch
    M, n = 2, 110
    mats = [synth.make_linear(3000 + i, 256, 256) + (256, 256) for i in range(n)]
    chain = [i > 0 and i % 2 == 0 for i in range(n)]
    x0 = synth.make_x(5, M, 256)
    outs, ads, xs = _oracle_chain(M, x0, mats, chain)
    ys = [torch.empty((M, 256), dtype=torch.float16, device="cuda") for _ in range(n)]
    ops = [((ys[i - 1] if chain[i] else to_dev(xs[i])), to_dev(qw), to_dev(s), to_dev(b), ys[i], chain[i])
           for i, (qw, s, b, _, _) in enumerate(mats)]
    w4.w4_gemv_seq(ops)
    torch.cuda.synchronize()
    for i in range(n):
        ok, worst = within_tol(ys[i].cpu().numpy(), outs[i], ads[i])
        assert ok, f"op {i}: worst err/tol = {worst}"


def test_seq_full_size_layer_sampled(w4):
    """One 3B layer's blocks (q|k|v, o, gate|up, down) at full size, independent
    activations; sampled rows against the oracle."""
    import torch
    M = 1
    plan = [(2048, 2560), (2048, 2048), (2048, 22016), (11008, 2048)]
    ops, refs = [], []
    g = np.random.default_rng(3)
    for i, (K, N) in enumerate(plan):
        qw, s, b = synth.make_linear(4100 + i, N, K)
        x = synth.make_x(4200 + i, M, K)
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        ops.append((to_dev(x), to_dev(qw), to_dev(s), to_dev(b), y, False))
        refs.append((x, qw, s, b, N, K, y))
    w4.w4_gemv_seq(ops)
    torch.cuda.synchronize()
    for x, qw, s, b, N, K, y in refs:
        rows = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 64)])).astype(np.int32)
        yo, ad = oracle.gemv_rows(x, qw, s, b, K, rows)
        ok, worst = within_tol(y.cpu().numpy()[:, rows], yo, ad)
        assert ok, worst


def test_seq_rejects_bad_arguments(w4):
    import ctypes
    import torch
    op = w4.GemvOp(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 64, 320, 0, 0)   # K % 256 != 0
    arr = (w4.GemvOp * 1)(op)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert w4.lib.w4_gemv_seq(ctypes.cast(arr, ctypes.c_void_p), 1, 1, ws.data_ptr(), 16, 0, None) == 2
    assert w4.lib.w4_gemv_seq(ctypes.cast(arr, ctypes.c_void_p), 1, 1, ws.data_ptr(), 8, 0, None) == 6
