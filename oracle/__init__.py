"""CPU oracle for GGUF block-quantized matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
library (``gguf_block_quantized_qmatmul_gb300``) never imports it and shares no
code with it: the arithmetic lives in ``qmm_oracle.c`` (plain C, compiled with
``-O2 -ffp-contract=off``), written from the candle tutorial pages
("同一个 GGUF，CPU 和 Metal 生成的文字不一样" section 出处; "自己量化" sections 3,
和下载的 Q8_0 逐字节比 and 大小和误差).  This module only marshals numpy arrays.

Parity status: every function is pinned by ``tests/test_oracle_pins.py`` except
the Q4_K, Q4_0, Q5_0 and Q6_K quantizers' choice of codes, which is "parity
unpinned" beyond their round-trip error bounds and closed forms (the pages give
neither the algorithms nor the Q4_0/Q5_0/Q6_K layouts, only their sizes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q8_0, Q4_K, Q8_K, Q4_0, Q5_0, Q6_K = 1, 2, 3, 4, 5, 6
NAMES = {"q8_0": Q8_0, "q4_k": Q4_K, "q8_k": Q8_K, "q4_0": Q4_0, "q5_0": Q5_0, "q6_k": Q6_K}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -ffast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
               "-std=gnu11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f32.restype = ctypes.c_float
            lib.orc_f32_to_f16_array.argtypes = [p, i64, p]
            lib.orc_f16_to_f32_array.argtypes = [p, i64, p]
            lib.orc_f16_check_range.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.orc_f16_check_range.restype = i64
            lib.orc_block_values.argtypes = [ctypes.c_int]
            lib.orc_block_values.restype = i64
            lib.orc_block_bytes.argtypes = [ctypes.c_int]
            lib.orc_block_bytes.restype = i64
            for f in ("orc_quantize_q8_0", "orc_quantize_q8_k", "orc_quantize_q4_k", "orc_quantize_q4_0",
                      "orc_quantize_q5_0", "orc_quantize_q6_k"):
                getattr(lib, f).argtypes = [p, i64, i64, p]
            lib.orc_dequantize.argtypes = [ctypes.c_int, p, i64, i64, p]
            lib.orc_block_sums.argtypes = [ctypes.c_int, p, p, i64, i64, i64, p]
            lib.orc_matmul_int8_act.argtypes = [ctypes.c_int, p, p, i64, i64, i64, p, p]
            lib.orc_matmul_f32_act.argtypes = [ctypes.c_int, p, p, i64, i64, i64, p, p]
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _t(t) -> int:
    return NAMES[t] if isinstance(t, str) else int(t)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32)


def block_values(t) -> int:
    return int(_load().orc_block_values(_t(t)))


def block_bytes(t) -> int:
    return int(_load().orc_block_bytes(_t(t)))


def row_bytes(t, K: int) -> int:
    bv = block_values(t)
    if K % bv:
        raise ValueError(f"K={K} is not a multiple of the block size {bv}")
    return K // bv * block_bytes(t)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (n <= 0: all available); the
    results do not depend on it."""
    _load().orc_set_num_threads(int(n))


def f32_to_f16_bits(x) -> np.ndarray:
    x = _f32(x).ravel()
    out = np.empty(x.size, dtype=np.uint16)
    _load().orc_f32_to_f16_array(_ptr(x), x.size, _ptr(out))
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.empty(h.size, dtype=np.float32)
    _load().orc_f16_to_f32_array(_ptr(h), h.size, _ptr(out))
    return out


def f16_check_range(lo: int, hi: int) -> int:
    """Mismatches of the oracle's f32->f16 against the compiler's _Float16 cast."""
    return int(_load().orc_f16_check_range(lo, hi))


def quantize(t, x) -> np.ndarray:
    """Quantize rows of x [rows, K] to blocks; returns uint8 [rows, row_bytes]."""
    x = _f32(x)
    if x.ndim == 1:
        x = x[None, :]
    rows, K = x.shape
    out = np.empty((rows, row_bytes(t, K)), dtype=np.uint8)
    fn = {Q8_0: "orc_quantize_q8_0", Q8_K: "orc_quantize_q8_k", Q4_K: "orc_quantize_q4_k",
          Q4_0: "orc_quantize_q4_0", Q5_0: "orc_quantize_q5_0", Q6_K: "orc_quantize_q6_k"}[_t(t)]
    getattr(_load(), fn)(_ptr(x), rows, K, _ptr(out))
    return out


def dequantize(t, q, K: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows = q.size // row_bytes(t, K)
    out = np.empty((rows, K), dtype=np.float32)
    _load().orc_dequantize(_t(t), _ptr(q), rows, K, _ptr(out))
    return out


def block_sums(wtype, wq, xq, M: int, N: int, K: int) -> np.ndarray:
    """Exact per-block integer sums.  Q8_0, Q4_0, Q5_0 (with Q8_0 activations):
    int32 [M, N, K/32]; Q4_K: int32 [M, N, K/256, 2] holding (S_sc, S_m);
    Q6_K: int32 [M, N, K/256] holding S = sum_j sc_j isum_j."""
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    if _t(wtype) == Q4_K:
        out = np.empty((M, N, K // 256, 2), dtype=np.int32)
    elif _t(wtype) == Q6_K:
        out = np.empty((M, N, K // 256), dtype=np.int32)
    else:
        out = np.empty((M, N, K // 32), dtype=np.int32)
    _load().orc_block_sums(_t(wtype), _ptr(wq), _ptr(xq), M, N, K, _ptr(out))
    return out


def matmul(wtype, mode: str, wq, x):
    """y [M, N] (float64) and the tolerance scale T [M, N] (sum of |terms|).

    mode "int8_act": activations quantized per row (Q8_0 for Q8_0, Q4_0 and
    Q5_0 weights; Q8K for Q4_K and Q6_K), integer
    block sums, float combine.  mode "f32_act": f32 activations times the
    dequantized weights (equal by definition to the dequantize-all form)."""
    x = _f32(x)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    N = wq.size // row_bytes(wtype, K)
    y = np.empty((M, N), dtype=np.float64)
    T = np.empty((M, N), dtype=np.float64)
    fn = {"int8_act": "orc_matmul_int8_act", "f32_act": "orc_matmul_f32_act"}[mode]
    getattr(_load(), fn)(_t(wtype), _ptr(wq), _ptr(x), M, N, K, _ptr(y), _ptr(T))
    return y, T


def tolerance(T):
    """Per-element float bound: |y_gpu - y_oracle| <= 1e-5 * T + 1e-6."""
    return 1e-5 * np.asarray(T) + 1e-6
