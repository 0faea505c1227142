"""GB300-native (sm_103a) int4 weight-only affine linear layer (W4A16).

Thin Python binding of ``libw4a16.so``: every function here validates and
marshals torch tensors into the C ABI declared in ``include/w4a16.h`` and
enqueues the library's CUDA kernels on the current torch stream.  There is no
CPU or PyTorch fallback: if the library is missing, importing this package
fails.

Weight format: ``qweight`` int32/uint32 [N][K/8] (8 four-bit codes per word,
lowest nibble = lowest k), ``scales`` and ``biases`` float16 [N][K/group]
(group 64 unless given); w[n][k] = scale * q + bias, or, with
``biases=None``, symmetric codes w[n][k] = scale * (q - 8).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["OVERLAP_PREVIOUS", "w4_gemv", "w4_gemv_seq", "GemvList", "seq_workspace", "seq_workspace_bytes", "GemvOp",
           "lm_head_argmax_topk", "lm_head_workspace_bytes", "w4_dequant_f16", "f16_gemm", "w4_gemm",
           "w4_gemm_workspace", "w4_gemm_workspace_bytes", "device_status", "W4A16Error", "LIB_PATH", "lib"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")

STATUS = {0: "W4A16_OK", 1: "W4_ERR_NULL", 2: "W4_ERR_SHAPE", 3: "W4_ERR_ALIGN", 4: "W4_ERR_GROUP",
          5: "W4_ERR_LAUNCH", 6: "W4_ERR_WORKSPACE", 7: "W4_ERR_DEVICE", 8: "W4_ERR_TIMEOUT"}


class W4A16Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} "
                         f"({lib.w4a16_status_string(status).decode()})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                          "(nvcc, sm_103a) before importing this package")
    L = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.w4_gemv.argtypes = [P, P, P, P, P, I, I, I, I, P]
    L.lm_head_argmax_topk.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P, Z, P]
    L.w4_gemv_ex.argtypes = [P, P, P, P, P, I, I, I, I, ctypes.c_uint, P]
    L.lm_head_argmax_topk_ex.argtypes = [P, P, P, P, I, I, I, I, I, P, P, P, Z, ctypes.c_uint, P]
    L.w4_gemv_seq.argtypes = [P, I, I, P, Z, ctypes.c_uint, P]
    L.w4_gemv_seq_workspace_bytes.argtypes = []
    L.w4_gemv_seq_workspace_bytes.restype = Z
    L.w4_gemv_seq_workspace_bytes_ex.argtypes = [P, I, I]
    L.w4_gemv_seq_workspace_bytes_ex.restype = Z
    L.lm_head_workspace_bytes.argtypes = [I, I, I]
    L.lm_head_workspace_bytes.restype = Z
    L.w4_dequant_f16.argtypes = [P, P, P, P, I, I, I, P]
    L.w4_dequant_f16_ex.argtypes = [P, P, P, P, I, I, I, ctypes.c_uint, P]
    L.f16_gemm.argtypes = [P, P, P, I, I, I, P]
    L.w4_gemm.argtypes = [P, P, P, P, P, I, I, I, I, P, Z, P]
    L.w4_gemm_ex.argtypes = [P, P, P, P, P, I, I, I, I, P, Z, ctypes.c_uint, P]
    L.w4_gemm_workspace_bytes.argtypes = [I, I, I]
    L.w4_gemm_workspace_bytes.restype = Z
    L.f16_gemm_ex.argtypes = [P, P, P, I, I, I, ctypes.c_uint, P]
    L.w4a16_status_string.argtypes = [I]
    L.w4a16_status_string.restype = ctypes.c_char_p
    L.w4a16_device_status.argtypes = []
    for f in ("w4_gemv", "w4_gemv_ex", "w4_gemv_seq", "lm_head_argmax_topk", "lm_head_argmax_topk_ex",
              "w4_dequant_f16", "w4_dequant_f16_ex", "f16_gemm", "f16_gemm_ex", "w4a16_device_status"):
        getattr(L, f).restype = I
    return L


lib = _load()


def _check(fn: str, status: int):
    if status != 0:
        raise W4A16Error(fn, status)


def _dev(t: torch.Tensor, name: str, dtypes) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


_QW = (torch.int32, getattr(torch, "uint32", torch.int32))
OVERLAP_PREVIOUS = 1  # W4A16_OVERLAP_PREVIOUS: stream weights before the previous kernel finishes
_H = (torch.float16,)


def _weight_dims(qweight, scales, biases, group):
    N, KW = qweight.shape
    K = KW * 8
    if group < 1 or K % group != 0:
        raise ValueError(f"group {group} does not divide K = {K}")
    if scales.shape != (N, K // group) or (biases is not None and biases.shape != (N, K // group)):
        raise ValueError(f"scales/biases must be [{N}][{K // group}]")
    return N, K


def _biases(b) -> int | None:
    """Device pointer of the biases, or NULL (None) for symmetric codes."""
    return None if b is None else _dev(b, "biases", _H)


def w4_gemv(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
            y: torch.Tensor | None = None, group: int = 64, stream=None, flags: int = 0) -> torch.Tensor:
    """y[M][N] = x[M][K] @ W^T for the int4 weight (M <= 16).  flags: 0 or
    OVERLAP_PREVIOUS (the weights must not be written by the previous kernel)."""
    N, K = _weight_dims(qweight, scales, biases, group)
    x2 = x.reshape(-1, K) if x.dim() != 2 else x
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check("w4_gemv", lib.w4_gemv_ex(_dev(x2, "x", _H), _dev(qweight, "qweight", _QW),
                                     _dev(scales, "scales", _H), _biases(biases),
                                     _dev(y, "y", _H), M, N, K, group, flags, _stream(stream)))
    return y


class GemvOp(ctypes.Structure):
    """One operation of w4_gemv_seq (mirror of the C struct w4_gemv_op)."""
    _fields_ = [("x", ctypes.c_void_p), ("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("wait_prev", ctypes.c_int), ("group", ctypes.c_int)]


def _seq_array(ops, group):
    arr = (GemvOp * len(ops))()
    M = None
    for i, op in enumerate(ops):
        x, qw, s, b, y, wait = op[:6]
        g = op[6] if len(op) > 6 else group
        N, K = _weight_dims(qw, s, b, g)
        x2 = x.reshape(-1, K) if x.dim() != 2 else x
        if M is None:
            M = x2.shape[0]
        elif x2.shape[0] != M:
            raise ValueError("all operations must have the same number of activation rows")
        arr[i] = GemvOp(_dev(x2, "x", _H), _dev(qw, "qweight", _QW), _dev(s, "scales", _H),
                        _biases(b), _dev(y, "y", _H), N, K, 1 if wait else 0, g)
    return arr, M


def seq_workspace_bytes(ops, group: int = 64) -> int:
    """Workspace bytes for w4_gemv_seq(ops) with the tagged activation exchange
    (w4_gemv_seq_workspace_bytes_ex); a smaller workspace of at least
    w4_gemv_seq_workspace_bytes() bytes selects the completion-counter path."""
    arr, M = _seq_array(ops, group)
    return int(lib.w4_gemv_seq_workspace_bytes_ex(ctypes.cast(arr, ctypes.c_void_p), len(ops), M))


def seq_workspace(ops, group: int = 64) -> torch.Tensor:
    """A zero-filled workspace for w4_gemv_seq(ops); reuse it for every later
    call with the same list (its counters reset themselves)."""
    return torch.zeros(seq_workspace_bytes(ops, group), dtype=torch.uint8, device=ops[0][0].device)


class GemvList:
    """A projection list checked and marshalled once, for calling w4_gemv_seq
    every decode step: run() only hands the prepared operation array to the
    library, which in turn reuses its launch plan for an unchanged list.  The
    tensors of `ops` (see w4_gemv_seq) are kept referenced by this object."""

    def __init__(self, ops, group: int = 64):
        self.ops = list(ops)
        self.arr, self.M = _seq_array(self.ops, group)
        self.ptr = ctypes.cast(self.arr, ctypes.c_void_p)
        self.nops = len(self.ops)

    def workspace_bytes(self) -> int:
        return int(lib.w4_gemv_seq_workspace_bytes_ex(self.ptr, self.nops, self.M))

    def workspace(self) -> torch.Tensor:
        """A zero-filled workspace for this list (reuse it for every call)."""
        return torch.zeros(self.workspace_bytes(), dtype=torch.uint8, device=self.ops[0][0].device)

    def run(self, workspace: torch.Tensor, stream=None):
        _check("w4_gemv_seq", lib.w4_gemv_seq(self.ptr, self.nops, self.M,
                                              _dev(workspace, "workspace", (torch.uint8,)), workspace.numel(),
                                              0, _stream(stream)))
        return [op[4] for op in self.ops]


def w4_gemv_seq(ops, workspace: torch.Tensor | None = None, group: int = 64, stream=None):
    """Run a list of GEMVs in one persistent launch.

    ops: a GemvList, or a sequence of (x, qweight, scales, biases, y,
    wait_prev[, group]) with torch tensors (biases None: symmetric codes);
    wait_prev = True when x is written by an earlier operation of the list;
    group defaults to `group`.  All x share the same number of rows M.
    workspace: from seq_workspace(ops) (zero-filled before its first use,
    then passed unchanged to every call); a fresh one is made when None.
    Returns the list of y."""
    gl = ops if isinstance(ops, GemvList) else GemvList(ops, group)
    if workspace is None:
        workspace = gl.workspace()
    return gl.run(workspace, stream)


def lm_head_workspace_bytes(M: int, N: int, k: int) -> int:
    return int(lib.lm_head_workspace_bytes(M, N, k))


def lm_head_argmax_topk(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                        biases: torch.Tensor, k: int = 1, idx: torch.Tensor | None = None,
                        val: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        group: int = 64, stream=None, flags: int = 0):
    """(idx int32 [M][k], val float32 [M][k]): the k largest logits of x @ W^T per row."""
    N, K = _weight_dims(qweight, scales, biases, group)
    x2 = x.reshape(-1, K) if x.dim() != 2 else x
    M = x2.shape[0]
    if idx is None:
        idx = torch.empty((M, k), dtype=torch.int32, device=x.device)
    if val is None:
        val = torch.empty((M, k), dtype=torch.float32, device=x.device)
    need = lm_head_workspace_bytes(M, N, k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check("lm_head_argmax_topk",
           lib.lm_head_argmax_topk_ex(_dev(x2, "x", _H), _dev(qweight, "qweight", _QW),
                                      _dev(scales, "scales", _H), _biases(biases),
                                      M, N, K, group, k, _dev(idx, "idx", (torch.int32,)),
                                      _dev(val, "val", (torch.float32,)),
                                      _dev(workspace, "workspace", (torch.uint8,)),
                                      workspace.numel(), flags, _stream(stream)))
    return idx, val


def w4_dequant_f16(qweight: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor,
                   w16: torch.Tensor | None = None, group: int = 64, stream=None, flags: int = 0) -> torch.Tensor:
    """Transposed half scratch w16[K][N] = RNE(scale * q + bias), or
    RNE(scale * (q - 8)) with biases None.  flags:
    OVERLAP_PREVIOUS when this call shares no memory with the previous kernel
    (it may then run concurrently with it)."""
    N, K = _weight_dims(qweight, scales, biases, group)
    if w16 is None:
        w16 = torch.empty((K, N), dtype=torch.float16, device=qweight.device)
    _check("w4_dequant_f16",
           lib.w4_dequant_f16_ex(_dev(qweight, "qweight", _QW), _dev(scales, "scales", _H),
                                 _biases(biases), _dev(w16, "w16", _H), N, K, group, flags,
                                 _stream(stream)))
    return w16


def w4_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib.w4_gemm_workspace_bytes(M, N, K))


def w4_gemm_workspace(M: int, N: int, K: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for w4_gemm at these sizes (reusable by every
    later call with sizes that need no more)."""
    return torch.zeros(max(w4_gemm_workspace_bytes(M, N, K), 16), dtype=torch.uint8, device=device or "cuda")


def w4_gemm(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor | None,
            y: torch.Tensor | None = None, group: int = 64, workspace: torch.Tensor | None = None, stream=None,
            flags: int = 0) -> torch.Tensor:
    """y[M][N] = x[M][K] @ W^T with the int4 weight dequantised inside the
    tensor-core GEMM (M <= 128).  workspace: from w4_gemm_workspace (zero-filled
    once, then reused); a fresh one is made when None."""
    N, K = _weight_dims(qweight, scales, biases, group)
    x2 = x.reshape(-1, K) if x.dim() != 2 else x
    M = x2.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if workspace is None:
        workspace = w4_gemm_workspace(M, N, K, x.device)
    _check("w4_gemm", lib.w4_gemm_ex(_dev(x2, "x", _H), _dev(qweight, "qweight", _QW), _dev(scales, "scales", _H),
                                     _biases(biases), _dev(y, "y", _H), M, N, K, group,
                                     _dev(workspace, "workspace", (torch.uint8,)), workspace.numel(), flags,
                                     _stream(stream)))
    return y


def f16_gemm(x16: torch.Tensor, w16: torch.Tensor, y: torch.Tensor | None = None,
             stream=None, flags: int = 0) -> torch.Tensor:
    """y[M][N] = x16[M][K] @ w16[K][N] (fp32 accumulation, half output).  flags:
    OVERLAP_PREVIOUS when w16 is complete before the previous kernel on the
    stream started (the kernel then fetches it early and waits only before x16
    and y)."""
    M, K = x16.shape
    K2, N = w16.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x16.device)
    _check("f16_gemm", lib.f16_gemm_ex(_dev(x16, "x16", _H), _dev(w16, "w16", _H), _dev(y, "y", _H),
                                       M, N, K, flags, _stream(stream)))
    return y


def device_status() -> int:
    """Synchronise and return the library's device-side status (0 = ok, 8 = a bounded wait expired)."""
    return int(lib.w4a16_device_status())
