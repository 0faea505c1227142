"""The C-ABI library loads, exports every function include/w4a16.h declares,
and rejects bad arguments on the host (no CUDA call is made on these paths)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "w4a16.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))
LIB = os.path.join(ROOT, "int4_weight_only_affine_gb300", "libw4a16.so")


def _declared():
    names = []
    for h in HEADERS:
        names += re.findall(r"W4A16_API\s+[\w\s\*]+?\b(\w+)\s*\(", open(h).read())
    return names


def _status_codes():
    text = open(HEADER).read()
    return {m[0]: int(m[1]) for m in re.findall(r"#define\s+(W4\w+)\s+(\d+)", text)}


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_hot_path_calls():
    names = set(_declared())
    assert {"w4_gemv", "w4_gemv_ex", "w4_gemv_seq", "w4_gemv_seq_workspace_bytes", "w4_gemv_seq_workspace_bytes_ex",
            "lm_head_argmax_topk", "lm_head_argmax_topk_ex", "lm_head_argmax_topk_noalloc",
            "lm_head_workspace_bytes", "w4_dequant_f16", "w4_dequant_f16_ex", "f16_gemm", "f16_gemm_ex",
            "w4_gemm", "w4_gemm_ex", "w4_gemm_workspace_bytes", "w4a16_status_string",
            "w4a16_device_status", "w4a16_testing_set_seq_wait"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def _args(lib):
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.w4_gemv.argtypes = [P, P, P, P, P, I, I, I, I, P]
    lib.lm_head_argmax_topk.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P, Z, P]
    lib.lm_head_workspace_bytes.argtypes = [I, I, I]
    lib.lm_head_workspace_bytes.restype = Z
    lib.w4_dequant_f16.argtypes = [P, P, P, P, I, I, I, P]
    lib.f16_gemm.argtypes = [P, P, P, I, I, I, P]
    lib.w4a16_status_string.argtypes = [I]
    lib.w4a16_status_string.restype = ctypes.c_char_p
    return lib


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case below fails a host check first


def test_host_validation_codes(lib):
    L = _args(lib)
    c = _status_codes()
    f = FAKE
    # w4_gemv
    assert L.w4_gemv(None, f, f, f, f, 1, 8, 64, 64, None) == c["W4_ERR_NULL"]
    assert L.w4_gemv(f, f, f, f, None, 1, 8, 64, 64, None) == c["W4_ERR_NULL"]
    assert L.w4_gemv(f, None, f, f, f, 1, 8, 64, 64, None) == c["W4_ERR_NULL"]
    assert L.w4_gemv(f, f, None, f, f, 1, 8, 64, 64, None) == c["W4_ERR_NULL"]
    for bad in (0, -64, 16, 48, 96, 128):  # not a power of two in 32..K, or above K = 64
        assert L.w4_gemv(f, f, f, f, f, 1, 8, 64, bad, None) == c["W4_ERR_GROUP"], bad
        assert L.w4_gemv(f, f, f, None, f, 1, 8, 64, bad, None) == c["W4_ERR_GROUP"], bad
    assert L.w4_gemv(f, f, f, f, f, 1, 8, 192, 128, None) == c["W4_ERR_GROUP"]  # 192 % 128 != 0
    assert L.w4_gemv(f, f, f, f + 8, f, 1, 8, 64, 64, None) == c["W4_ERR_ALIGN"]
    assert L.w4_gemv(f, f, f, f, f, 0, 8, 64, 64, None) == c["W4_ERR_SHAPE"]
    assert L.w4_gemv(f, f, f, f, f, 17, 8, 64, 64, None) == c["W4_ERR_SHAPE"]
    assert L.w4_gemv(f, f, f, f, f, 1, 0, 64, 64, None) == c["W4_ERR_SHAPE"]
    assert L.w4_gemv(f, f, f, f, f, 1, 8, 96, 64, None) == c["W4_ERR_SHAPE"]
    assert L.w4_gemv(f + 8, f, f, f, f, 1, 8, 64, 64, None) == c["W4_ERR_ALIGN"]
    assert L.w4_gemv(f, f, f, f, f + 2, 1, 8, 64, 64, None) == c["W4_ERR_ALIGN"]
    # lm_head_argmax_topk
    need = L.lm_head_workspace_bytes(1, 1000, 5)
    assert need > 0
    assert L.lm_head_argmax_topk(f, f, f, f, 1, 1000, 64, 64, 5, f, f, None, need, None) == c["W4_ERR_WORKSPACE"]
    assert L.lm_head_argmax_topk(f, f, f, f, 1, 1000, 64, 64, 5, f, f, f, need - 1, None) == c["W4_ERR_WORKSPACE"]
    assert L.lm_head_argmax_topk(f, f, f, f, 1, 1000, 64, 64, 0, f, f, f, need, None) == c["W4_ERR_SHAPE"]
    assert L.lm_head_argmax_topk(f, f, f, f, 1, 1000, 64, 64, 65, f, f, f, 1 << 30, None) == c["W4_ERR_SHAPE"]
    assert L.lm_head_argmax_topk(f, f, f, f, 1, 4, 64, 64, 5, f, f, f, 1 << 30, None) == c["W4_ERR_SHAPE"]
    assert L.lm_head_argmax_topk(f, f, f, f, 1, 1000, 64, 64, 5, None, f, f, need, None) == c["W4_ERR_NULL"]
    assert L.lm_head_argmax_topk(f, f, f, f, 1, 1000, 64, 48, 5, f, f, f, need, None) == c["W4_ERR_GROUP"]
    # w4_dequant_f16
    assert L.w4_dequant_f16(f, f, f, None, 8, 64, 64, None) == c["W4_ERR_NULL"]
    assert L.w4_dequant_f16(f, f, f, f, 8, 100, 64, None) == c["W4_ERR_SHAPE"]
    assert L.w4_dequant_f16(f, f, f, f, 8, 64, 128, None) == c["W4_ERR_GROUP"]
    assert L.w4_dequant_f16(f, None, f, f, 8, 64, 64, None) == c["W4_ERR_NULL"]
    assert L.w4_dequant_f16(f, f, None, f, 8, 128, 96, None) == c["W4_ERR_GROUP"]
    assert L.w4_dequant_f16(f, f, None, f, 8, 128, 256, None) == c["W4_ERR_GROUP"]
    assert L.w4_dequant_f16(f, f + 4, f, f, 8, 64, 64, None) == c["W4_ERR_ALIGN"]
    # f16_gemm
    assert L.f16_gemm(None, f, f, 4, 8, 8, None) == c["W4_ERR_NULL"]
    assert L.f16_gemm(f, f, f, 4, 12, 8, None) == c["W4_ERR_SHAPE"]
    assert L.f16_gemm(f, f, f, 0, 8, 8, None) == c["W4_ERR_SHAPE"]
    assert L.f16_gemm(f, f, f, 4, 8, 4, None) == c["W4_ERR_SHAPE"]
    assert L.f16_gemm(f, f + 8, f, 4, 8, 8, None) == c["W4_ERR_ALIGN"]


def test_workspace_bytes_formula(lib):
    L = _args(lib)
    # M * min(ceil(N/16), 16384 // k) * k * 8 bytes of candidate keys
    assert L.lm_head_workspace_bytes(1, 151936, 1) == 1 * 9496 * 1 * 8
    assert L.lm_head_workspace_bytes(1, 151936, 50) == 1 * (16384 // 50) * 50 * 8
    assert L.lm_head_workspace_bytes(16, 1000, 5) == 16 * 63 * 5 * 8
    assert L.lm_head_workspace_bytes(0, 1000, 5) == 0
    assert L.lm_head_workspace_bytes(1, 1000, 65) == 0
    assert L.lm_head_workspace_bytes(1, 4, 5) == 0


def test_status_strings(lib):
    L = _args(lib)
    for name, code in _status_codes().items():
        s = L.w4a16_status_string(code)
        assert s and s != b"unknown status", name
    assert L.w4a16_status_string(999) == b"unknown status"


class _Op(ctypes.Structure):
    """Mirror of w4_gemv_op (the C struct of include/w4a16.h)."""
    _fields_ = [("x", ctypes.c_void_p), ("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("wait_prev", ctypes.c_int), ("group", ctypes.c_int)]


def _seq_bytes(lib, ops, M):
    lib.w4_gemv_seq_workspace_bytes_ex.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    lib.w4_gemv_seq_workspace_bytes_ex.restype = ctypes.c_size_t
    arr = (_Op * len(ops))(*ops)
    return lib.w4_gemv_seq_workspace_bytes_ex(ctypes.cast(arr, ctypes.c_void_p), len(ops), M)


def test_seq_workspace_sizes_follow_the_producer_of_each_input(lib):
    """Host-only: the tagged-exchange workspace holds one uint32 per output
    element of each operation whose output a later waiting operation reads
    (x inside that output: whole, prefix or interior), on top of the 16-byte
    counter head.  Addresses are never dereferenced."""
    lib.w4_gemv_seq_workspace_bytes.restype = ctypes.c_size_t
    head = lib.w4_gemv_seq_workspace_bytes()
    assert head == 16
    W = 0x7000_0000
    a, b, c, d = 0x1000_0000, 0x2000_0000, 0x3000_0000, 0x4000_0000
    M = 2
    # op1 reads all of op0's output, op2 reads a prefix of op1's, op3 reads an
    # unrelated buffer (counter path), op4 does not wait.
    ops = [_Op(a, W, W, W, b, 2560, 2048, 0, 0),
           _Op(b, W, W, W, c, 1024, 2560, 1, 0),
           _Op(c, W, W, W, d, 256, 512, 1, 0),
           _Op(a, W, W, W, d + 0x10_0000, 256, 2048, 1, 0),
           _Op(d, W, W, W, d + 0x20_0000, 256, 256, 0, 0)]
    want = head + M * 2560 * 4 + M * 1024 * 4
    assert _seq_bytes(lib, ops, M) == want
    # x straddling the end of the producer's output: counter path, no tagged copy
    ops2 = [_Op(a, W, W, W, b, 256, 256, 0, 0), _Op(b + 256, W, W, W, c, 256, 256, 1, 0)]
    assert _seq_bytes(lib, ops2, M) == head
    # a later writer of the same range shadows the earlier one
    ops3 = [_Op(a, W, W, W, b, 512, 256, 0, 0), _Op(a, W, W, W, b, 256, 256, 0, 0),
            _Op(b, W, W, W, c, 256, 256, 1, 0)]
    assert _seq_bytes(lib, ops3, 1) == head + 256 * 4


def test_seq_lists_split_by_scale_layout_class(lib):
    """Host-only: a launch runs operations of one scale-layout class (group-64
    affine, symmetric group 128, group 32, any other layout: one kernel
    variant each), so an
    activation exchange between classes needs no tagged copy (stream order
    covers it); within a run of one class it does."""
    lib.w4_gemv_seq_workspace_bytes.restype = ctypes.c_size_t
    head = lib.w4_gemv_seq_workspace_bytes()
    W = 0x7000_0000
    a, b, c = 0x1000_0000, 0x2000_0000, 0x3000_0000
    mixed = [_Op(a, W, W, W, b, 512, 256, 0, 64), _Op(b, W, W, 0, c, 256, 512, 1, 32)]
    assert _seq_bytes(lib, mixed, 1) == head
    same = [_Op(a, W, W, W, b, 512, 256, 0, 32), _Op(b, W, W, 0, c, 256, 512, 1, 32)]
    assert _seq_bytes(lib, same, 1) == head + 512 * 4
    default = [_Op(a, W, W, W, b, 512, 256, 0, 0), _Op(b, W, W, W, c, 256, 512, 1, 64)]
    assert _seq_bytes(lib, default, 2) == head + 2 * 512 * 4
    sym_after_affine = [_Op(a, W, W, W, b, 512, 256, 0, 0), _Op(b, W, W, 0, c, 256, 512, 1, 128)]
    assert _seq_bytes(lib, sym_after_affine, 2) == head
    other = [_Op(a, W, W, W, b, 512, 256, 0, 128), _Op(b, W, W, 0, c, 256, 512, 1, 256)]
    assert _seq_bytes(lib, other, 2) == head + 2 * 512 * 4
    sym128 = [_Op(a, W, W, 0, b, 512, 256, 0, 128), _Op(b, W, W, 0, c, 256, 512, 1, 128)]
    assert _seq_bytes(lib, sym128, 2) == head + 2 * 512 * 4
    sym128_then_other = [_Op(a, W, W, 0, b, 512, 256, 0, 128), _Op(b, W, W, W, c, 256, 512, 1, 128)]
    assert _seq_bytes(lib, sym128_then_other, 2) == head


def test_seq_rejects_bad_operation_groups(lib):
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.w4_gemv_seq.argtypes = [P, I, I, P, Z, ctypes.c_uint, P]
    c = _status_codes()
    f = FAKE
    for bad in (-1, 16, 48, 512):
        ops = (_Op * 1)(_Op(f, f, f, f, f, 64, 256, 0, bad))
        assert lib.w4_gemv_seq(ctypes.cast(ops, P), 1, 1, f, 16, 0, None) == c["W4_ERR_GROUP"], bad


def test_w4_gemm_host_validation(lib):
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.w4_gemm.argtypes = [P, P, P, P, P, I, I, I, I, P, Z, P]
    lib.w4_gemm_workspace_bytes.argtypes = [I, I, I]
    lib.w4_gemm_workspace_bytes.restype = Z
    c = _status_codes()
    f = FAKE
    need = lib.w4_gemm_workspace_bytes(64, 256, 512)
    # counters (256 bytes) + 512 slot flags + 256 tile counters + two fp32
    # partial tiles (M x 128) per CTA for at most min(256, tiles x k steps)
    # = 2 x 8 = 16 CTAs
    assert need == 3328 + 2 * 16 * 64 * 128 * 4
    # the CTA count is capped at 256 whatever the size
    assert lib.w4_gemm_workspace_bytes(128, 22016, 2048) == 3328 + 2 * 256 * 128 * 128 * 4
    assert lib.w4_gemm_workspace_bytes(129, 256, 512) == 0
    assert lib.w4_gemm_workspace_bytes(4, 12, 512) == 0
    assert lib.w4_gemm_workspace_bytes(4, 256, 96) == 0
    g = lib.w4_gemm
    assert g(None, f, f, f, f, 64, 256, 512, 64, f, need, None) == c["W4_ERR_NULL"]
    assert g(f, f, None, f, f, 64, 256, 512, 64, f, need, None) == c["W4_ERR_NULL"]
    assert g(f, f, f, f, None, 64, 256, 512, 64, f, need, None) == c["W4_ERR_NULL"]
    assert g(f, f, f, f, f, 0, 256, 512, 64, f, need, None) == c["W4_ERR_SHAPE"]
    assert g(f, f, f, f, f, 129, 256, 512, 64, f, need, None) == c["W4_ERR_SHAPE"]
    assert g(f, f, f, f, f, 64, 12, 512, 64, f, need, None) == c["W4_ERR_SHAPE"]
    assert g(f, f, f, f, f, 64, 256, 96, 32, f, need, None) == c["W4_ERR_SHAPE"]
    assert g(f, f, f, f, f, 64, 256, 512, 48, f, need, None) == c["W4_ERR_GROUP"]
    assert g(f, f, f, None, f, 64, 256, 512, 1024, f, need, None) == c["W4_ERR_GROUP"]
    assert g(f, f, f, f, f, 64, 256, 512, 64, None, need, None) == c["W4_ERR_WORKSPACE"]
    assert g(f, f, f, f, f, 64, 256, 512, 64, f, need - 1, None) == c["W4_ERR_WORKSPACE"]
    assert g(f + 8, f, f, f, f, 64, 256, 512, 64, f, need, None) == c["W4_ERR_ALIGN"]
    assert g(f, f, f, f, f, 64, 256, 512, 64, f + 4, need, None) == c["W4_ERR_ALIGN"]
    lib.w4_gemm_ex.argtypes = [P, P, P, P, P, I, I, I, I, P, Z, ctypes.c_uint, P]
    for bad_flags in (2, 0x80000000):
        assert lib.w4_gemm_ex(f, f, f, f, f, 64, 256, 512, 64, f, need, bad_flags, None) == c["W4_ERR_SHAPE"]
