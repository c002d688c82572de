"""ORACLE -- test infrastructure only (tests, smoke check, benchmark CPU baseline).

Python view of ``oracle.c``: a plain fp64 CPU statement of the activation quantizer, the block decoders
and the GEMV / W8A16 products.  It shares no code with the CUDA library and is never imported by it.
"""
import ctypes
import os

import numpy as np

from . import _build

Q4_K, Q6_K, Q8_0, Q5_K = 1, 2, 3, 5
FMT = {"Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K, "Q8_0": Q8_0}
_lib = None


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB_OVERRIDE loads another build of oracle.c (the mutation test plants mistakes in copies)
        L = ctypes.CDLL(os.environ.get("ORACLE_LIB_OVERRIDE") or _build.build())
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.oracle_fp16_to_f64.restype = ctypes.c_double
        L.oracle_fp16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f64.restype = ctypes.c_double
        L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_f32_to_fp16.restype = ctypes.c_uint16
        L.oracle_f32_to_fp16.argtypes = [ctypes.c_float]
        L.oracle_quantize_act.restype = None
        L.oracle_quantize_act.argtypes = [vp, i32, i32, vp]
        L.oracle_dequant_q8_1.restype = None
        L.oracle_dequant_q8_1.argtypes = [vp, i32, i32, vp]
        L.oracle_row_bytes.restype = i64
        L.oracle_row_bytes.argtypes = [i32, i32]
        L.oracle_dequant_row.restype = i32
        L.oracle_dequant_row.argtypes = [i32, vp, i32, i64, vp]
        L.oracle_gemv_rows.restype = i32
        L.oracle_gemv_rows.argtypes = [i32, vp, vp, i32, i32, i32, vp, i64, vp]
        L.oracle_w8a16_rows.restype = i32
        L.oracle_w8c_rows.restype = i32
        L.oracle_w8c_rows.argtypes = [vp, vp, vp, i32, i32, i32, vp, i64, vp]
        L.oracle_w8a16_rows.argtypes = [vp, vp, i32, i32, i32, vp, i64, vp]
        _lib = L
    return _lib


def _fmt(fmt):
    return FMT[fmt] if isinstance(fmt, str) else int(fmt)


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def fp16_to_f64(h: int) -> float:
    return lib().oracle_fp16_to_f64(int(h) & 0xFFFF)


def bf16_to_f64(b: int) -> float:
    return lib().oracle_bf16_to_f64(int(b) & 0xFFFF)


def f32_to_fp16(f: float) -> int:
    return lib().oracle_f32_to_fp16(ctypes.c_float(np.float32(f)))


def quantize_act(x: np.ndarray) -> np.ndarray:
    """fp32 [m, K] -> q8_1 bytes [m, K/32 * 36]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    m, K = x.shape
    assert K % 32 == 0
    out = np.empty((m, K // 32 * 36), dtype=np.uint8)
    lib().oracle_quantize_act(_ptr(x), m, K, _ptr(out))
    return out


def widen16(kind: str, x16: np.ndarray) -> np.ndarray:
    """bf16 or binary16 bit patterns -> fp32 values (exact: both types are subsets of binary32)."""
    dec = bf16_to_f64 if kind == "bf16" else fp16_to_f64
    flat = np.ascontiguousarray(x16, dtype=np.uint16).reshape(-1)
    return np.array([dec(int(v)) for v in flat], dtype=np.float32).reshape(np.shape(x16))


def quantize_act16(kind: str, x16: np.ndarray) -> np.ndarray:
    """The q8_1 quantizer on 16-bit activation rows: widen to fp32, then the fp32 definition."""
    return quantize_act(widen16(kind, x16))


def dequant_act(xq: np.ndarray, m: int, K: int) -> np.ndarray:
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    out = np.empty((m, K), dtype=np.float64)
    lib().oracle_dequant_q8_1(_ptr(xq), m, K, _ptr(out))
    return out


def row_bytes(fmt, K: int) -> int:
    return int(lib().oracle_row_bytes(_fmt(fmt), K))


def dequant_rows(fmt, W: np.ndarray, N: int, K: int, rows=None) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    rows = range(N) if rows is None else rows
    out = np.empty((len(rows), K), dtype=np.float64)
    for r, n in enumerate(rows):
        rc = lib().oracle_dequant_row(_fmt(fmt), _ptr(W), K, int(n), ctypes.c_void_p(out[r].ctypes.data))
        assert rc == 0
    return out


def gemv(fmt, W: np.ndarray, xq: np.ndarray, m: int, N: int, K: int, rows=None) -> np.ndarray:
    """y [m, len(rows)] (fp64); rows=None means all N rows."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    if rows is None:
        rp, nr = None, N
    else:
        ra = np.ascontiguousarray(rows, dtype=np.int64)
        rp, nr = _ptr(ra), len(ra)
    y = np.empty((m, nr), dtype=np.float64)
    rc = lib().oracle_gemv_rows(_fmt(fmt), _ptr(W), _ptr(xq), m, N, K, rp, nr, _ptr(y))
    assert rc == 0, rc
    return y


def w8a16(W: np.ndarray, x_bf16: np.ndarray, m: int, N: int, K: int, rows=None) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if rows is None:
        rp, nr = None, N
    else:
        ra = np.ascontiguousarray(rows, dtype=np.int64)
        rp, nr = _ptr(ra), len(ra)
    y = np.empty((m, nr), dtype=np.float64)
    rc = lib().oracle_w8a16_rows(_ptr(W), _ptr(x), m, N, K, rp, nr, _ptr(y))
    assert rc == 0, rc
    return y


def w8a16_channel(Wq: np.ndarray, scale: np.ndarray, x_bf16: np.ndarray, m: int, N: int, K: int,
                  rows=None) -> np.ndarray:
    """Per-channel INT8 weights int8 [N, K], fp32 scales [N], bf16 activations [m, K] -> y [m, len(rows)]."""
    Wq = np.ascontiguousarray(Wq).view(np.int8).reshape(-1)
    sc = np.ascontiguousarray(scale, dtype=np.float32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if rows is None:
        rp, nr = None, N
    else:
        ra = np.ascontiguousarray(rows, dtype=np.int64)
        rp, nr = _ptr(ra), len(ra)
    y = np.empty((m, nr), dtype=np.float64)
    rc = lib().oracle_w8c_rows(_ptr(Wq), _ptr(sc), _ptr(x), m, N, K, rp, nr, _ptr(y))
    assert rc == 0, rc
    return y
