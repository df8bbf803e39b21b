"""GGUF block-quantized matmul for GB300 (sm_103a): thin Python binding.

Every computation runs in the CUDA library ``_build/libqmm.so`` through its C
ABI (``include/qmm.h``); this module only marshals torch tensors (device
pointers, sizes, the current CUDA stream) and raises on error statuses.  There
is no CPU fallback: the first call raises ImportError when the library is
missing.

Entry points mirror the C ABI names:
  quantize_weights(w, wtype)      Q8_0 / Q4_K / Q4_0 / Q5_0 / Q6_K blocks of f32 weights [N, K]
  quantize_act(x, atype)          Q8_0 / Q8_K blocks of f32 activations [M, K]
  dequantize(q, t, K)             f32 [rows, K]
  matmul(wq, x, wtype, mode)      y = x . W^T, mode "int8_act" or "f32_act"
  block_sums(wq, x, wtype)        exact per-block integer sums of the int8_act form
  matmul_batch(items, wtype, mode)  many independent small matmuls in one launch
  matmul_batch_typed(items, mode)   the same, each item with its own weight type
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

QMM_F32, QMM_Q8_0, QMM_Q4_K, QMM_Q8_K, QMM_Q4_0, QMM_Q5_0, QMM_Q6_K = 0, 1, 2, 3, 4, 5, 6
QMM_INT8_ACT, QMM_F32_ACT = 0, 1
TYPES = {"f32": QMM_F32, "q8_0": QMM_Q8_0, "q4_k": QMM_Q4_K, "q8_k": QMM_Q8_K, "q4_0": QMM_Q4_0, "q5_0": QMM_Q5_0,
         "q6_k": QMM_Q6_K}
MODES = {"int8_act": QMM_INT8_ACT, "f32_act": QMM_F32_ACT}
STATUS = {0: "QMM_OK", 1: "QMM_ERR_NULL", 2: "QMM_ERR_SHAPE", 3: "QMM_ERR_TYPE", 4: "QMM_ERR_ALIGN",
          5: "QMM_ERR_WORKSPACE", 6: "QMM_ERR_CUDA", 7: "QMM_ERR_TIMEOUT"}

# every symbol declared in include/qmm.h
EXPORTS = ["qmm_block_values", "qmm_block_bytes", "qmm_row_bytes", "qmm_quantize_weights", "qmm_quantize_act",
           "qmm_dequantize", "qmm_matmul_workspace", "qmm_matmul_launches", "qmm_matmul", "qmm_matmul_static_workspace",
           "qmm_block_sums", "qmm_matmul_batch", "qmm_matmul_batch_typed", "qmm_test_inject", "qmm_test_set_wait_limit",
           "qmm_last_device_error", "qmm_status_string"]
INJECT = {"off": 0, "launch_failure": 1, "stall": 2}


class QmmError(RuntimeError):
    def __init__(self, status: int, call: str, text: str):
        super().__init__(f"{call}: {STATUS.get(status, status)} ({text})")
        self.status = status


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libqmm.so is not built ({path}); run __graft_entry__.build() or "
                          f"python -m gguf_block_quantized_qmatmul_gb300.build")
    lib = ctypes.CDLL(path)
    i64, sz, p, i32 = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
    lib.qmm_block_values.argtypes, lib.qmm_block_values.restype = [i32], i64
    lib.qmm_block_bytes.argtypes, lib.qmm_block_bytes.restype = [i32], sz
    lib.qmm_row_bytes.argtypes, lib.qmm_row_bytes.restype = [i32, i64], sz
    lib.qmm_quantize_weights.argtypes, lib.qmm_quantize_weights.restype = [i32, p, i64, i64, p, p], i32
    lib.qmm_quantize_act.argtypes, lib.qmm_quantize_act.restype = [i32, p, i64, i64, p, p], i32
    lib.qmm_dequantize.argtypes, lib.qmm_dequantize.restype = [i32, p, i64, i64, p, p], i32
    lib.qmm_matmul_workspace.argtypes, lib.qmm_matmul_workspace.restype = [i32, i32, i64, i64, i64], sz
    lib.qmm_matmul_launches.argtypes, lib.qmm_matmul_launches.restype = [i32, i32, i64, i64, i64], i32
    lib.qmm_matmul.argtypes, lib.qmm_matmul.restype = [i32, i32, p, p, p, i64, i64, i64, p, sz, p], i32
    lib.qmm_block_sums.argtypes, lib.qmm_block_sums.restype = [i32, p, p, i64, i64, i64, p, p], i32
    lib.qmm_matmul_batch.argtypes, lib.qmm_matmul_batch.restype = [i32, i32, p, i64, p], i32
    lib.qmm_matmul_batch_typed.argtypes, lib.qmm_matmul_batch_typed.restype = [i32, p, i64, p], i32
    lib.qmm_test_inject.argtypes, lib.qmm_test_inject.restype = [i32, i32, i32], i32
    lib.qmm_test_set_wait_limit.argtypes, lib.qmm_test_set_wait_limit.restype = [i32], i32
    lib.qmm_last_device_error.argtypes, lib.qmm_last_device_error.restype = [], i32
    lib.qmm_status_string.argtypes, lib.qmm_status_string.restype = [i32], ctypes.c_char_p
    return lib


_LIB = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def _t(t) -> int:
    return TYPES[t] if isinstance(t, str) else int(t)


def _m(m) -> int:
    return MODES[m] if isinstance(m, str) else int(m)


def _check(status: int, call: str) -> None:
    if status != 0:
        raise QmmError(status, call, _lib().qmm_status_string(status).decode())


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def block_values(t) -> int:
    return int(_lib().qmm_block_values(_t(t)))


def block_bytes(t) -> int:
    return int(_lib().qmm_block_bytes(_t(t)))


def row_bytes(t, K: int) -> int:
    return int(_lib().qmm_row_bytes(_t(t), K))


def quantize_weights(w: torch.Tensor, wtype, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    N, K = w.shape
    if out is None:
        out = torch.empty((N, row_bytes(wtype, K)), dtype=torch.uint8, device=w.device)
    _check(_lib().qmm_quantize_weights(_t(wtype), _ptr(w), N, K, _ptr(out), _stream(stream)), "qmm_quantize_weights")
    return out


def quantize_act(x: torch.Tensor, atype, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    M, K = x.shape
    if out is None:
        out = torch.empty((M, row_bytes(atype, K)), dtype=torch.uint8, device=x.device)
    _check(_lib().qmm_quantize_act(_t(atype), _ptr(x), M, K, _ptr(out), _stream(stream)), "qmm_quantize_act")
    return out


def dequantize(q: torch.Tensor, t, K: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rb = row_bytes(t, K)
    rows = q.numel() // rb if rb else 0
    if out is None:
        out = torch.empty((rows, K), dtype=torch.float32, device=q.device)
    _check(_lib().qmm_dequantize(_t(t), _ptr(q), rows, K, _ptr(out), _stream(stream)), "qmm_dequantize")
    return out


def matmul_workspace(wtype, mode, M: int, N: int, K: int) -> int:
    return int(_lib().qmm_matmul_workspace(_t(wtype), _m(mode), M, N, K))


def matmul_launches(wtype, mode, M: int, N: int, K: int) -> int:
    """Kernel launches of one matmul call for this shape (a diagnostic)."""
    return int(_lib().qmm_matmul_launches(_t(wtype), _m(mode), M, N, K))


def matmul(wq: torch.Tensor, x: torch.Tensor, wtype, mode, N: int | None = None, out: torch.Tensor | None = None,
           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    M, K = x.shape
    if N is None:
        N = wq.numel() // row_bytes(wtype, K)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if workspace is None:  # a caller's workspace is checked by the library (QMM_ERR_WORKSPACE)
        need = matmul_workspace(wtype, mode, M, N, K)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().qmm_matmul(_t(wtype), _m(mode), _ptr(wq), _ptr(x), _ptr(out), M, N, K, _ptr(workspace), ws_bytes,
                          _stream(stream)), "qmm_matmul")
    return out


def block_sums(wq: torch.Tensor, x: torch.Tensor, wtype, N: int | None = None, stream=None) -> torch.Tensor:
    M, K = x.shape
    if N is None:
        N = wq.numel() // row_bytes(wtype, K)
    if _t(wtype) == QMM_Q4_K:  # (S_sc, S_m) per super-block
        out = torch.empty((M, N, K // 256, 2), dtype=torch.int32, device=x.device)
    elif _t(wtype) == QMM_Q6_K:  # S per super-block
        out = torch.empty((M, N, K // 256), dtype=torch.int32, device=x.device)
    else:  # 32-value blocks (Q8_0, Q4_0, Q5_0)
        out = torch.empty((M, N, K // 32), dtype=torch.int32, device=x.device)
    _check(_lib().qmm_block_sums(_t(wtype), _ptr(wq), _ptr(x), M, N, K, _ptr(out), _stream(stream)), "qmm_block_sums")
    return out


class MatmulDesc(ctypes.Structure):
    """qmm_matmul_desc: one item of qmm_matmul_batch."""
    _fields_ = [("wq", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class MatmulBatch:
    """A descriptor table for qmm_matmul_batch, built once: items are (wq, x,
    y) device tensors, y [M, N] receiving x . W^T.  run() launches it (one
    launch per 256 items; the table travels in the launch parameters)."""

    def __init__(self, items, wtype, mode):
        self.items = list(items)  # keeps the tensors alive
        self.wtype, self.mode = _t(wtype), _m(mode)
        self.descs = (MatmulDesc * max(len(self.items), 1))()
        for i, (wq, x, y) in enumerate(self.items):
            M, K = x.shape
            self.descs[i] = MatmulDesc(_ptr(wq), _ptr(x), _ptr(y), M, y.shape[1], K)
        self.ptr = ctypes.cast(self.descs, ctypes.c_void_p)

    def run(self, stream=None):
        _check(_lib().qmm_matmul_batch(self.wtype, self.mode, self.ptr, len(self.items), _stream(stream)),
               "qmm_matmul_batch")


def matmul_batch(items, wtype, mode, stream=None):
    """One-off qmm_matmul_batch over (wq, x, y) items; returns the ys."""
    b = MatmulBatch(items, wtype, mode)
    b.run(stream)
    return [y for _, _, y in b.items]


class TypedMatmulDesc(ctypes.Structure):
    """qmm_matmul_typed_desc: one item of qmm_matmul_batch_typed."""
    _fields_ = [("wtype", ctypes.c_int), ("wq", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class MatmulBatchTyped:
    """A descriptor table for qmm_matmul_batch_typed, built once: items are
    (wtype, wq, x, y), each with its own weight type (a decode step of a
    mixed-type file); run() launches it (one launch per 256 items)."""

    def __init__(self, items, mode):
        self.items = list(items)  # keeps the tensors alive
        self.mode = _m(mode)
        self.descs = (TypedMatmulDesc * max(len(self.items), 1))()
        for i, (t, wq, x, y) in enumerate(self.items):
            M, K = x.shape
            self.descs[i] = TypedMatmulDesc(_t(t), _ptr(wq), _ptr(x), _ptr(y), M, y.shape[1], K)
        self.ptr = ctypes.cast(self.descs, ctypes.c_void_p)

    def run(self, stream=None):
        _check(_lib().qmm_matmul_batch_typed(self.mode, self.ptr, len(self.items), _stream(stream)),
               "qmm_matmul_batch_typed")


def matmul_batch_typed(items, mode, stream=None):
    """One-off qmm_matmul_batch_typed over (wtype, wq, x, y) items; returns the ys."""
    b = MatmulBatchTyped(items, mode)
    b.run(stream)
    return [y for _, _, _, y in b.items]


def last_device_error() -> int:
    return int(_lib().qmm_last_device_error())


def test_inject(kind: str, count: int = 1, arg: int = 0) -> None:
    """Failure-test hook: arm an injected failure ("launch_failure": the next
    `count` matmul calls return QMM_ERR_CUDA without touching the device;
    "stall": the next decode-kernel launch withholds its first block's weight
    stages from stage `arg` on, so a bounded wait times out; "off")."""
    _check(_lib().qmm_test_inject(INJECT[kind], count, arg), "qmm_test_inject")


def test_set_wait_limit(log2_clocks: int) -> None:
    """Failure-test hook: spin limit of the device's bounded waits, 2^log2
    SM clocks (0 restores the default of about one second)."""
    _check(_lib().qmm_test_set_wait_limit(log2_clocks), "qmm_test_set_wait_limit")
