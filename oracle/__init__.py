"""CPU oracle for the row softmax -- TEST INFRASTRUCTURE ONLY.

A plain double-precision C implementation of the softmax definition
(``oracle_softmax.c``), loaded with ctypes.  Only the tests, the smoke check
and the bench's CPU-baseline leg use it; the GPU library never imports it and
the two share no code.  Every function cites the passage it follows in the C
source.

Inputs are the storage arrays of ``memory_bound_row_softmax_gb300.workloads``:
float32 for f32, raw uint16 bit patterns for f16 and bf16, shape
``(rows, row_stride)``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_softmax.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_softmax.so")
_DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/liboracle_softmax.so``."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.POINTER(ctypes.c_double)
            lib.oracle_softmax_rows.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int]
            lib.oracle_softmax_rows.restype = ctypes.c_int
            lib.oracle_softmax_masked_rows.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int,
                                                       ctypes.c_double, i64, i64]
            lib.oracle_softmax_masked_rows.restype = ctypes.c_int
            lib.oracle_attention_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_int, ctypes.c_double,
                                                 ctypes.c_int, i64]
            lib.oracle_attention_fwd.restype = ctypes.c_int
            lib.oracle_row_stats.argtypes = [vp, i64, i64, i64, i64, ctypes.c_int, vp]
            lib.oracle_online_stats.argtypes = [vp, i64, vp, i64, i64, ctypes.c_int, vp]
            lib.oracle_merge.argtypes = [ctypes.c_double] * 4 + [dp, dp]
            lib.oracle_merge.restype = None
            lib.oracle_tree_merge.argtypes = [vp, vp, i64, vp]
            lib.oracle_tree_merge.restype = ctypes.c_int
            lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_f16.restype = ctypes.c_double
            lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_bf16.restype = ctypes.c_double
            _lib = lib
    return _lib


def _check_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    want = np.float32 if dtype == "f32" else np.uint16
    if x.dtype != want or x.ndim != 2:
        raise TypeError(f"oracle wants a 2-D {np.dtype(want).name} array for {dtype}, got {x.dtype} {x.shape}")
    return np.ascontiguousarray(x)


def softmax(x: np.ndarray, dtype: str, cols: int | None = None, rows=None, threads: int = 1) -> np.ndarray:
    """Row softmax in double precision (definition: max, shifted exp, sum, divide).

    ``x`` is a (R, row_stride) storage array; the first ``cols`` columns are valid
    (default: all).  ``rows`` selects a subset of row indices (default: all).
    Returns float64 of shape (len(rows), cols).  ``threads`` > 1 splits the rows
    over a thread pool (ctypes releases the GIL while the C code runs).
    """
    lib = _load()
    x = _check_storage(x, dtype)
    stride = x.shape[1]
    cols = stride if cols is None else cols
    code = _DTYPE_CODE[dtype]
    if rows is None:
        sel = None
        nrows = x.shape[0]
    else:
        sel = np.asarray(rows, dtype=np.int64)
        nrows = len(sel)
    out = np.empty((nrows, cols), dtype=np.float64)
    if nrows == 0:
        return out

    def run(lo: int, hi: int):
        scratch = np.empty(cols, dtype=np.float64)
        if sel is None:
            rc = lib.oracle_softmax_rows(x.ctypes.data, out[lo:hi].ctypes.data, scratch.ctypes.data,
                                         lo, hi, cols, stride, code)
            assert rc == 0
        else:
            for i in range(lo, hi):
                r = int(sel[i])
                rc = lib.oracle_softmax_rows(x.ctypes.data, out[i:i + 1].ctypes.data, scratch.ctypes.data,
                                             r, r + 1, cols, stride, code)
                assert rc == 0

    if threads <= 1 or nrows < 2:
        run(0, nrows)
    else:
        step = (nrows + threads - 1) // threads
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda lo: run(lo, min(nrows, lo + step)), range(0, nrows, step)))
    return out


def softmax_masked(x: np.ndarray, dtype: str, scale: float, causal_offset: int, rows_per_seq: int = 0,
                   cols: int | None = None, rows=None, threads: int = 1) -> np.ndarray:
    """Scaled, causally masked row softmax in double precision: row r keeps
    columns c <= (r mod rows_per_seq) + causal_offset (rows_per_seq <= 0: r
    itself), scaled by ``scale``; masked outputs are 0 and masked inputs are
    never read; a row that keeps nothing is NaN.  Arguments as ``softmax``."""
    lib = _load()
    x = _check_storage(x, dtype)
    stride = x.shape[1]
    cols = stride if cols is None else cols
    code = _DTYPE_CODE[dtype]
    sel = np.arange(x.shape[0], dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    nrows = len(sel)
    out = np.empty((nrows, cols), dtype=np.float64)
    if nrows == 0:
        return out

    def run(lo: int, hi: int):
        scratch = np.empty(cols, dtype=np.float64)
        if rows is None:
            rc = lib.oracle_softmax_masked_rows(x.ctypes.data, out[lo:hi].ctypes.data, scratch.ctypes.data, lo, hi,
                                                cols, stride, code, float(scale), causal_offset, rows_per_seq)
            assert rc == 0
        else:
            for i in range(lo, hi):
                r = int(sel[i])
                rc = lib.oracle_softmax_masked_rows(x.ctypes.data, out[i:i + 1].ctypes.data, scratch.ctypes.data,
                                                    r, r + 1, cols, stride, code, float(scale), causal_offset,
                                                    rows_per_seq)
                assert rc == 0

    if threads <= 1 or nrows < 2:
        run(0, nrows)
    else:
        step = (nrows + threads - 1) // threads
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda lo: run(lo, min(nrows, lo + step)), range(0, nrows, step)))
    return out


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, dtype: str, scale: float, causal: bool = False,
                  causal_offset: int = 0) -> np.ndarray:
    """One head of attention in double precision: O = softmax(Q K^T * scale,
    causal mask keeping key j <= query i + causal_offset) V.  q: (n_q, d),
    k, v: (n_k, d) storage arrays of ``dtype``; returns float64 (n_q, d)."""
    lib = _load()
    q, k, v = (_check_storage(a, dtype) for a in (q, k, v))
    if k.shape != v.shape or q.shape[1] != k.shape[1]:
        raise ValueError(f"shapes q {q.shape}, k {k.shape}, v {v.shape} do not fit")
    n_q, d = q.shape
    out = np.empty((n_q, d), dtype=np.float64)
    scratch = np.empty(k.shape[0], dtype=np.float64)
    rc = lib.oracle_attention_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data, scratch.ctypes.data,
                                  n_q, k.shape[0], d, _DTYPE_CODE[dtype], float(scale), 1 if causal else 0,
                                  causal_offset)
    assert rc == 0
    return out


def row_stats(x: np.ndarray, dtype: str, row: int, c_begin: int, c_end: int) -> tuple[float, float]:
    """(m, l) of columns [c_begin, c_end) of one row, taken directly."""
    lib = _load()
    x = _check_storage(x, dtype)
    s = np.empty(2, dtype=np.float64)
    lib.oracle_row_stats(x.ctypes.data, row, c_begin, c_end, x.shape[1], _DTYPE_CODE[dtype], s.ctypes.data)
    return float(s[0]), float(s[1])


def online_stats(x: np.ndarray, dtype: str, row: int, bounds) -> tuple[float, float]:
    """(m, l) of one row folded chunk by chunk with the two-state merge rule."""
    lib = _load()
    x = _check_storage(x, dtype)
    b = np.ascontiguousarray(bounds, dtype=np.int64)
    s = np.empty(2, dtype=np.float64)
    lib.oracle_online_stats(x.ctypes.data, row, b.ctypes.data, len(b), x.shape[1], _DTYPE_CODE[dtype],
                            s.ctypes.data)
    return float(s[0]), float(s[1])


def merge(m1: float, l1: float, m2: float, l2: float) -> tuple[float, float]:
    """The two-state merge: m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m)."""
    lib = _load()
    m, l = ctypes.c_double(), ctypes.c_double()
    lib.oracle_merge(m1, l1, m2, l2, ctypes.byref(m), ctypes.byref(l))
    return m.value, l.value


def tree_merge(m, l):
    """Stride-halving merge tree; returns (m, l, per-round surviving maxima)."""
    lib = _load()
    m = np.ascontiguousarray(m, dtype=np.float64).copy()
    l = np.ascontiguousarray(l, dtype=np.float64).copy()
    n = len(m)
    trace = np.empty(max(1, n), dtype=np.float64)
    rc = lib.oracle_tree_merge(m.ctypes.data, l.ctypes.data, n, trace.ctypes.data)
    if rc != 0:
        raise ValueError("tree_merge needs a power-of-two count")
    rounds, t, s = [], 0, n // 2
    while s > 0:
        rounds.append(trace[t:t + s].tolist())
        t += s
        s //= 2
    return float(m[0]), float(l[0]), rounds


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode f16/bf16 bit patterns to float64 with the oracle's own decoder."""
    lib = _load()
    f = lib.oracle_decode_f16 if dtype == "f16" else lib.oracle_decode_bf16
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([f(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))
