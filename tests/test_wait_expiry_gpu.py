"""The failure path of the device-side bounded waits, driven without a fault.

Every wait inside the kernels is bounded; when one gives up, the kernel
records the expiry, lets its own copies land and returns, and
w4a16_device_status reports W4_ERR_TIMEOUT.  Here a test hook
(include/w4a16_testing.h) shortens the projection list's completion-counter
wait to 1 ms and raises its target past anything the list can reach, so the
wait cannot be met.  The call must return within a fraction of a second, the
status must say so exactly once, and the next normal call on a re-zeroed
workspace must again match the oracle.  Nothing traps, faults or hangs."""
import ctypes
import time

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
    w4.lib.w4a16_testing_set_seq_wait.argtypes = [ctypes.c_ulonglong, ctypes.c_uint]
    w4.lib.w4a16_testing_set_seq_wait.restype = ctypes.c_int
    return w4


def test_counter_wait_expiry_reports_timeout_and_recovers(w4):
    import torch
    M = 1
    plan = [(1024, 2048), (2048, 1024), (1024, 512)]   # (K, N); ops 1 and 2 read the previous output
    mats = [synth.make_linear(1500 + i, N, K) for i, (K, N) in enumerate(plan)]
    x0 = synth.make_x(1510, M, plan[0][0])
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _, N in plan]
    ops = [((ys[i - 1] if i else to_dev(x0)), to_dev(qw), to_dev(s), to_dev(b), ys[i], i > 0)
           for i, (qw, s, b) in enumerate(mats)]
    # A counters-only workspace: every wait of the list uses the completion counter.
    ws = torch.zeros(int(w4.lib.w4_gemv_seq_workspace_bytes()), dtype=torch.uint8, device="cuda")
    assert ws.numel() == 16
    assert w4.device_status() == 0
    assert w4.lib.w4a16_testing_set_seq_wait(3_000_000_000, 0) != 0   # above the 2 s ceiling
    try:
        assert w4.lib.w4a16_testing_set_seq_wait(1_000_000, 1) == 0  # 1 ms, unmeetable target
        t0 = time.perf_counter()
        w4.w4_gemv_seq(ops, workspace=ws)
        status = w4.device_status()   # synchronises
        elapsed = time.perf_counter() - t0
    finally:
        assert w4.lib.w4a16_testing_set_seq_wait(0, 0) == 0
    assert status == 8, w4.lib.w4a16_status_string(status)   # W4_ERR_TIMEOUT
    assert elapsed < 1.0, f"the expired wait took {elapsed:.3f} s (limit 1 ms, default 2 s)"
    assert w4.device_status() == 0   # the record is cleared once read

    # Normal operation again on a re-zeroed workspace: the oracle's chain.
    ws.zero_()
    w4.w4_gemv_seq(ops, workspace=ws)
    assert w4.device_status() == 0
    x = x0
    for i, ((qw, s, b), (K, N)) in enumerate(zip(mats, plan)):
        if i:
            x = oracle.double_to_half_array(y.ravel()).reshape(M, -1).view(np.float16)
        y, ad = oracle.gemv(x, qw, s, b, N, K, threads=16)
        ok, worst = within_tol(ys[i].cpu().numpy(), y, ad)
        assert ok, f"op {i}: worst err/tol = {worst}"
