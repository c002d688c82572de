"""Python binding of libqgemv (the C ABI declared in include/qgemv.h).

Argument marshalling only: every step of the quantizer and the GEMV runs in the CUDA kernels of
``libqgemv.so``.  Arguments may be torch tensors (their device pointer is passed) or raw integer device
addresses; ``stream`` may be a torch.cuda.Stream, a raw cudaStream_t integer, or None (torch's current
stream).  A non-zero status raises :class:`QgemvError`.  There is no fallback of any kind: if the
compiled library is missing, importing the binding's entry points raises.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqgemv.so")

QGEMV_Q4_K, QGEMV_Q6_K, QGEMV_Q8_0, QGEMV_W8A16, QGEMV_Q5_K, QGEMV_W8A16_CHANNEL = 1, 2, 3, 4, 5, 6
FMT = {"Q4_K": QGEMV_Q4_K, "Q5_K": QGEMV_Q5_K, "Q6_K": QGEMV_Q6_K, "Q8_0": QGEMV_Q8_0, "W8A16": QGEMV_W8A16,
       "W8A16_CHANNEL": QGEMV_W8A16_CHANNEL}
QGEMV_ACT_Q8_1, QGEMV_ACT_F32, QGEMV_ACT_BF16, QGEMV_ACT_F16 = 0, 1, 2, 3
ACT = {"q8_1": QGEMV_ACT_Q8_1, "f32": QGEMV_ACT_F32, "bf16": QGEMV_ACT_BF16, "f16": QGEMV_ACT_F16}
QGEMV_FLAG_PDL = 1
QGEMV_FLAG_PDL_LATE_TRIGGER = 2
QGEMV_MAX_GROUP = 8
QGEMV_ARGMAX_STATIC_SCRATCH_BYTES = 16384
ROUTE_FUSED, ROUTE_GROUPED, ROUTE_PDL, ROUTE_Q5_K_M1, ROUTE_W8A16_CHANNEL_M1, ROUTE_ARGMAX, ROUTE_M16 = (
    33, 34, 35, 36, 44, 52, 53)
ROUTE_CHUNKED = 54
STATUS = {0: "QGEMV_OK", 1: "QGEMV_ERR_INVALID_ARG", 2: "QGEMV_ERR_UNSUPPORTED", 3: "QGEMV_ERR_MISALIGNED",
          4: "QGEMV_ERR_CUDA", 5: "QGEMV_ERR_DEVICE", 6: "QGEMV_ERR_OVERLAP"}
NUM_ROUTES = 55

_lib = None


class QgemvMat(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int)]


class QgemvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS.get(status, f"status {status}")
        extra = ""
        if status == 4 and _lib is not None:
            extra = f" (cudaError {_lib.qgemv_last_cuda_error()})"
        super().__init__(f"{where}: {name}{extra}")


def lib():
    """Load libqgemv.so (built by ``build()``); raises if it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libqgemv.so not built at {LIB_PATH}; run quantized_weight_gemv_quantize_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.qgemv_quantize_act.argtypes = [vp, i32, i32, vp, vp]
        L.qgemv.argtypes = [i32, vp, vp, vp, i32, i32, i32, vp]
        L.qgemv_w8a16.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.qgemv_quantize_act_ex.argtypes = [vp, i32, i32, vp, ctypes.c_uint, vp]
        L.qgemv_quantize_act_typed.argtypes = [i32, vp, i32, i32, vp, ctypes.c_uint, vp]
        L.qgemv_w8a16_channel.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
        L.qgemv_w8a16_channel_ex.argtypes = [vp, vp, vp, vp, i32, i32, i32, ctypes.c_uint, vp]
        L.qgemv_max_k_w8a16_channel.argtypes = [i32]
        L.qgemv_max_k_w8a16_channel.restype = i32
        L.qgemv_tune_pairs.argtypes = [i32]
        L.qgemv_tune_pairs.restype = None
        L.qgemv_argmax_scratch_bytes.argtypes = [i32]
        L.qgemv_argmax_scratch_bytes.restype = sz
        L.qgemv_argmax.argtypes = [i32, vp, vp, i32, i32, i32, vp, sz, vp, vp, ctypes.c_uint, vp]
        L.qgemv_argmax.restype = i32
        L.qgemv_argmax_noalloc.argtypes = [i32, vp, vp, i32, i32, i32, vp, vp, ctypes.c_uint, vp]
        L.qgemv_argmax_noalloc.restype = i32
        L.qgemv_ex.argtypes = [i32, vp, vp, vp, i32, i32, i32, ctypes.c_uint, vp]
        L.qgemv_w8a16_ex.argtypes = [vp, vp, vp, i32, i32, i32, ctypes.c_uint, vp]
        L.qgemv_multi.argtypes = [i32, i32, ctypes.POINTER(QgemvMat), i32, vp, vp, i32, i32, ctypes.c_uint, vp]
        for f in ("qgemv_quantize_act", "qgemv", "qgemv_w8a16", "qgemv_quantize_act_ex", "qgemv_ex",
                  "qgemv_w8a16_ex", "qgemv_multi", "qgemv_quantize_act_typed", "qgemv_w8a16_channel",
                  "qgemv_w8a16_channel_ex"):
            getattr(L, f).restype = i32
        L.qgemv_weight_bytes.argtypes = [i32, i32, i32]
        L.qgemv_weight_bytes.restype = sz
        L.qgemv_act_bytes.argtypes = [i32, i32]
        L.qgemv_act_bytes.restype = sz
        L.qgemv_max_k.argtypes = [i32, i32]
        L.qgemv_max_k.restype = i32
        L.qgemv_max_k_w8a16.argtypes = [i32]
        L.qgemv_max_k_w8a16.restype = i32
        L.qgemv_chunk_k.argtypes = [i32, i32, i32]
        L.qgemv_chunk_k.restype = i32
        L.qgemv_status_string.argtypes = [i32]
        L.qgemv_status_string.restype = ctypes.c_char_p
        L.qgemv_last_cuda_error.argtypes = []
        L.qgemv_last_cuda_error.restype = i32
        L.qgemv_route_counts.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i32]
        L.qgemv_route_counts.restype = i32
        L.qgemv_route_reset.argtypes = []
        L.qgemv_route_reset.restype = None
        L.qgemv_debug_fail_next.argtypes = [i32, i32]
        L.qgemv_debug_fail_next.restype = None
        L.qgemv_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
        L.qgemv_device_error.restype = i32
        L.qgemv_plan_info.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_longlong)]
        L.qgemv_plan_info.restype = i32
        L.qgemv_plan_info_chunk.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_longlong)]
        L.qgemv_plan_info_chunk.restype = i32
        L.qgemv_tune_override.argtypes = [i32, i32, i32, i32, i32]
        L.qgemv_tune_override.restype = None
        ip = ctypes.POINTER(ctypes.c_int)
        L.qgemv_trace_info.argtypes = [ip, ip, ip]
        L.qgemv_trace_info.restype = i32
        L.qgemv_trace_begin.argtypes = []
        L.qgemv_trace_begin.restype = i32
        L.qgemv_trace_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), sz, ip]
        L.qgemv_trace_read.restype = i32
        _lib = L
    return _lib


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def use_trace_build() -> str:
    """Build the launch-timeline library (libqgemv_trace.so) and make it the one this process loads; must
    come before the first call that loads the library."""
    global LIB_PATH
    if _lib is not None:
        raise RuntimeError("use_trace_build() must come before the library is loaded")
    from . import _build
    LIB_PATH = _build.build(trace=True)
    return LIB_PATH


def trace_begin() -> None:
    _check(lib().qgemv_trace_begin(), "qgemv_trace_begin")


def trace_read():
    """The timeline records as a uint64 array [launches, ctas, fields] and the number of launches numbered."""
    import numpy as np
    nl, nc, nf = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().qgemv_trace_info(ctypes.byref(nl), ctypes.byref(nc), ctypes.byref(nf)), "qgemv_trace_info")
    buf = np.zeros(nl.value * nc.value * nf.value, dtype=np.uint64)
    n = ctypes.c_int()
    _check(lib().qgemv_trace_read(buf.ctypes.data_as(ctypes.POINTER(ctypes.c_ulonglong)), buf.nbytes,
                                  ctypes.byref(n)), "qgemv_trace_read")
    return buf.reshape(nl.value, nc.value, nf.value), n.value


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _fmt(fmt):
    return FMT[fmt] if isinstance(fmt, str) else int(fmt)


def _check(status: int, where: str):
    if status != 0:
        raise QgemvError(status, where)


def qgemv_quantize_act(x, m: int, K: int, xq, stream=None) -> None:
    _check(lib().qgemv_quantize_act(_ptr(x), m, K, _ptr(xq), _stream(stream)), "qgemv_quantize_act")


def qgemv(fmt, W, xq, y, m: int, N: int, K: int, stream=None) -> None:
    _check(lib().qgemv(_fmt(fmt), _ptr(W), _ptr(xq), _ptr(y), m, N, K, _stream(stream)), "qgemv")


def qgemv_w8a16(W, x_bf16, y, m: int, N: int, K: int, stream=None) -> None:
    _check(lib().qgemv_w8a16(_ptr(W), _ptr(x_bf16), _ptr(y), m, N, K, _stream(stream)), "qgemv_w8a16")


def qgemv_quantize_act_ex(x, m: int, K: int, xq, flags: int = 0, stream=None) -> None:
    _check(lib().qgemv_quantize_act_ex(_ptr(x), m, K, _ptr(xq), flags, _stream(stream)), "qgemv_quantize_act_ex")


def qgemv_quantize_act_typed(x_kind, x, m: int, K: int, xq, flags: int = 0, stream=None) -> None:
    """x_kind: "f32", "bf16", "f16" (or the QGEMV_ACT_* value); x holds m*K values of that kind."""
    xk = ACT[x_kind] if isinstance(x_kind, str) else int(x_kind)
    _check(lib().qgemv_quantize_act_typed(xk, _ptr(x), m, K, _ptr(xq), flags, _stream(stream)),
           "qgemv_quantize_act_typed")


def qgemv_w8a16_channel(Wq, scale, x_bf16, y, m: int, N: int, K: int, flags: int = 0, stream=None) -> None:
    """Per-output-channel INT8 weights (int8 [N, K]) with fp32 row scales [N] against bf16 [m, K]."""
    _check(lib().qgemv_w8a16_channel_ex(_ptr(Wq), _ptr(scale), _ptr(x_bf16), _ptr(y), m, N, K, flags,
                                        _stream(stream)), "qgemv_w8a16_channel")


def qgemv_argmax_scratch_bytes(m: int) -> int:
    return int(lib().qgemv_argmax_scratch_bytes(m))


def qgemv_argmax(fmt, W, xq, m: int, N: int, K: int, scratch, idx_out, val_out, flags: int = 0,
                 stream=None) -> None:
    """Fused GEMV + argmax: idx_out[i] / val_out[i] get the first row with the largest y[i, :]."""
    nbytes = scratch.numel() * scratch.element_size() if hasattr(scratch, "numel") else qgemv_argmax_scratch_bytes(m)
    _check(lib().qgemv_argmax(_fmt(fmt), _ptr(W), _ptr(xq), m, N, K, _ptr(scratch), nbytes, _ptr(idx_out),
                              _ptr(val_out), flags, _stream(stream)), "qgemv_argmax")


def qgemv_argmax_noalloc(fmt, W, xq, m: int, N: int, K: int, idx_out, val_out, flags: int = 0,
                         stream=None) -> None:
    """qgemv_argmax on the library's own static scratch (calls on a device must be ordered)."""
    _check(lib().qgemv_argmax_noalloc(_fmt(fmt), _ptr(W), _ptr(xq), m, N, K, _ptr(idx_out), _ptr(val_out), flags,
                                      _stream(stream)), "qgemv_argmax_noalloc")


def qgemv_max_k_w8a16_channel(m: int) -> int:
    return int(lib().qgemv_max_k_w8a16_channel(m))


def qgemv_ex(fmt, W, xq, y, m: int, N: int, K: int, flags: int = 0, stream=None) -> None:
    _check(lib().qgemv_ex(_fmt(fmt), _ptr(W), _ptr(xq), _ptr(y), m, N, K, flags, _stream(stream)), "qgemv_ex")


def qgemv_w8a16_ex(W, x_bf16, y, m: int, N: int, K: int, flags: int = 0, stream=None) -> None:
    _check(lib().qgemv_w8a16_ex(_ptr(W), _ptr(x_bf16), _ptr(y), m, N, K, flags, _stream(stream)), "qgemv_w8a16_ex")


def mats_array(mats):
    """[(W, y, N), ...] -> ctypes array of qgemv_mat (keep the result alive across the call)."""
    arr = (QgemvMat * len(mats))()
    for j, (W, y, N) in enumerate(mats):
        arr[j].W, arr[j].y, arr[j].N = _ptr(W), _ptr(y), int(N)
    return arr


def qgemv_multi(fmt, mats, act_kind, act, m: int, K: int, xq_out=None, flags: int = 0, stream=None) -> None:
    """mats: [(W, y, N), ...] sharing one activation; act_kind "q8_1" | "f32" | "bf16" (or its code)."""
    arr = mats if isinstance(mats, ctypes.Array) else mats_array(mats)
    kind = ACT[act_kind] if isinstance(act_kind, str) else int(act_kind)
    _check(lib().qgemv_multi(_fmt(fmt), len(arr), arr, kind, _ptr(act), _ptr(xq_out), m, K, flags,
                             _stream(stream)), "qgemv_multi")


def qgemv_weight_bytes(fmt, N: int, K: int) -> int:
    return int(lib().qgemv_weight_bytes(_fmt(fmt), N, K))


def qgemv_act_bytes(m: int, K: int) -> int:
    return int(lib().qgemv_act_bytes(m, K))


def qgemv_chunk_k(fmt, m: int, K: int) -> int:
    """Values per K-chunk of a call at (fmt, m, K): K when the rows take one pass of staging."""
    return int(lib().qgemv_chunk_k(_fmt(fmt), m, K))


def qgemv_max_k(fmt, m: int) -> int:
    return int(lib().qgemv_max_k(_fmt(fmt), m))


def qgemv_max_k_w8a16(m: int) -> int:
    return int(lib().qgemv_max_k_w8a16(m))


def qgemv_status_string(status: int) -> str:
    return lib().qgemv_status_string(status).decode()


def qgemv_route_counts():
    buf = (ctypes.c_ulonglong * NUM_ROUTES)()
    n = lib().qgemv_route_counts(buf, NUM_ROUTES)
    return [int(buf[i]) for i in range(min(n, NUM_ROUTES))]


def qgemv_route_reset() -> None:
    lib().qgemv_route_reset()


def qgemv_debug_fail_next(status: int, count: int = 1) -> None:
    lib().qgemv_debug_fail_next(status, count)


def qgemv_device_error(reset: bool = False) -> int:
    v = ctypes.c_uint(0)
    _check(lib().qgemv_device_error(ctypes.byref(v), 1 if reset else 0), "qgemv_device_error")
    return int(v.value)


PLAN_FIELDS = ("lanes", "rows_per_tile", "num_tiles", "stages", "stage_bytes", "smem", "grid", "row_bytes",
               "units_per_row", "x_stage_bytes", "threads", "team_warps", "red_bytes", "kernel_build")


def qgemv_plan_info(fmt, m: int, N: int, K: int, num_sms: int = 152, ctas_per_sm: int = 1) -> dict:
    """The launch plan for (fmt, m, N, K); fmt "W8A16" (or 4) asks for the W8A16 kernel."""
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    buf = (ctypes.c_longlong * 14)()
    _check(lib().qgemv_plan_info(f, m, N, K, num_sms, ctas_per_sm, buf), "qgemv_plan_info")
    return dict(zip(PLAN_FIELDS, [int(v) for v in buf]))


def qgemv_plan_info_chunk(fmt, m: int, N: int, Kc: int, num_sms: int = 152, ctas_per_sm: int = 1) -> dict:
    """The plan of one K-chunk launch of Kc values per row: qgemv_plan_info's fields plus slot_row_stride."""
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    buf = (ctypes.c_longlong * 15)()
    _check(lib().qgemv_plan_info_chunk(f, m, N, Kc, num_sms, ctas_per_sm, buf), "qgemv_plan_info_chunk")
    return dict(zip(PLAN_FIELDS + ("slot_row_stride",), [int(v) for v in buf]))


def qgemv_tune_pairs(mode: int = 0) -> None:
    """Tuning only: row pairs 0 = planner decides, 1 = whenever they fit, 2 = never."""
    lib().qgemv_tune_pairs(mode)


def qgemv_tune_override(ctas_per_sm: int = 0, lanes_log2: int = -1, rows_per_tile: int = 0, stages: int = 0,
                        kernel_build: int = 0) -> None:
    """Force plan parameters for sweeps (0 / -1 = planner decides).  Not for production use."""
    lib().qgemv_tune_override(ctas_per_sm, lanes_log2, rows_per_tile, stages, kernel_build)
