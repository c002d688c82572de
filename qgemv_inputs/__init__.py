"""Seeded synthetic inputs for the decode-GEMV workloads (shared by tests, benchmark and smoke check).

Holds only random-number generation and the storage layout of each block format (where a block's scale
bytes and code bytes sit); none of the quantize / dequantize / dot arithmetic.  Backed by ``gen.c``
(SplitMix64 in counter form), so every tensor is a pure function of its seed.
"""
import ctypes
import numpy as np

from . import _build
from .workloads import FORMATS, WORKLOADS, Workload, GemvOp, QuantOp  # noqa: F401

_lib = None

SCALE_LO = 1e-4
SCALE_HI = 1e-3


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u64, i64, vp, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.qgen_u64.restype = u64
        L.qgen_u64.argtypes = [u64, u64]
        L.qgen_derive.restype = u64
        L.qgen_derive.argtypes = [u64, u64]
        for name in ("qgen_q4k", "qgen_q5k", "qgen_q6k", "qgen_q80"):
            getattr(L, name).argtypes = [vp, i64, u64, dbl, dbl]
            getattr(L, name).restype = None
        for name in ("qgen_normal_f32", "qgen_normal_bf16", "qgen_bytes"):
            getattr(L, name).argtypes = [vp, i64, u64]
            getattr(L, name).restype = None
        L.qgen_fp16_uniform.argtypes = [vp, i64, u64, dbl, dbl]
        L.qgen_int8_sym.argtypes = [vp, i64, u64]
        L.qgen_int8_sym.restype = None
        L.qgen_f32_uniform.argtypes = [vp, i64, u64, dbl, dbl]
        L.qgen_f32_uniform.restype = None
        L.qgen_fp16_uniform.restype = None
        _lib = L
    return _lib


def u64(seed: int, counter: int) -> int:
    return lib().qgen_u64(seed & (2**64 - 1), counter & (2**64 - 1))


def derive(parent: int, *tags: int) -> int:
    s = parent & (2**64 - 1)
    for t in tags:
        s = lib().qgen_derive(s, t & (2**64 - 1))
    return s


def row_bytes(fmt: str, K: int) -> int:
    blk_bytes, blk_elems = FORMATS[fmt]
    assert K % blk_elems == 0, (fmt, K)
    return (K // blk_elems) * blk_bytes


def fill_weights_ptr(ptr: int, fmt: str, N: int, K: int, seed: int) -> None:
    """Fill host memory at ``ptr`` (N * row_bytes(fmt, K) bytes) with a seeded random matrix."""
    blk_bytes, blk_elems = FORMATS[fmt]
    nblocks = N * (K // blk_elems)
    fn = {"Q4_K": lib().qgen_q4k, "Q5_K": lib().qgen_q5k, "Q6_K": lib().qgen_q6k, "Q8_0": lib().qgen_q80}[fmt]
    fn(ctypes.c_void_p(ptr), nblocks, seed, SCALE_LO, SCALE_HI)


def weights(fmt: str, N: int, K: int, seed: int) -> np.ndarray:
    out = np.empty(N * row_bytes(fmt, K), dtype=np.uint8)
    fill_weights_ptr(out.ctypes.data, fmt, N, K, seed)
    return out


def fill_normal_f32_ptr(ptr: int, n: int, seed: int) -> None:
    assert n % 2 == 0
    lib().qgen_normal_f32(ctypes.c_void_p(ptr), n, seed)


def normal_f32(n: int, seed: int) -> np.ndarray:
    m = n + (n & 1)
    out = np.empty(m, dtype=np.float32)
    fill_normal_f32_ptr(out.ctypes.data, m, seed)
    return out[:n]


def fill_normal_bf16_ptr(ptr: int, n: int, seed: int) -> None:
    assert n % 2 == 0
    lib().qgen_normal_bf16(ctypes.c_void_p(ptr), n, seed)


def normal_bf16(n: int, seed: int) -> np.ndarray:
    """bf16 bit patterns (uint16) of RNE(fp32 N(0,1))."""
    m = n + (n & 1)
    out = np.empty(m, dtype=np.uint16)
    fill_normal_bf16_ptr(out.ctypes.data, m, seed)
    return out[:n]


def random_bytes(n: int, seed: int) -> np.ndarray:
    m = (n + 7) // 8 * 8
    out = np.empty(m, dtype=np.uint8)
    lib().qgen_bytes(ctypes.c_void_p(out.ctypes.data), m, seed)
    return out[:n]


def fp16_uniform(n: int, seed: int, lo: float = SCALE_LO, hi: float = SCALE_HI) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    lib().qgen_fp16_uniform(ctypes.c_void_p(out.ctypes.data), n, seed, lo, hi)
    return out


def channel_weights(N: int, K: int, seed: int):
    """Per-channel INT8 weights: (int8 [N*K] uniform -127..127, fp32 scales [N] uniform [SCALE_LO, SCALE_HI])."""
    w = np.empty(N * K, dtype=np.int8)
    lib().qgen_int8_sym(w.ctypes.data, N * K, seed)
    sc = np.empty(N, dtype=np.float32)
    lib().qgen_f32_uniform(sc.ctypes.data, N, derive(seed, 0x5CA1E), SCALE_LO, SCALE_HI)
    return w, sc
