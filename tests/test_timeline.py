"""The launch-timeline build (libqgemv_trace.so): the normal library answers the trace calls with
QGEMV_ERR_UNSUPPORTED; the traced library computes the same bits as the normal one and records every CTA of
every launch in order (entry <= dependency released <= activation staged <= done)."""
import ctypes

import numpy as np
import pytest

import qgemv_inputs as gen
import quantized_weight_gemv_quantize_gb300 as qg


@pytest.fixture(scope="module")
def L():
    qg.build()
    return qg.lib()


def test_normal_build_does_not_trace(L):
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert L.qgemv_trace_info(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) == 2
    assert L.qgemv_trace_begin() == 2
    buf = (ctypes.c_ulonglong * 4)()
    assert L.qgemv_trace_read(buf, 32, ctypes.byref(a)) == 2


@pytest.mark.gpu
def test_traced_build_records_every_cta_and_computes_the_same_bits(L):
    torch = pytest.importorskip("torch")
    from quantized_weight_gemv_quantize_gb300 import _build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    T = ctypes.CDLL(_build.build(trace=True))
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    T.qgemv_quantize_act_ex.argtypes = [vp, i32, i32, vp, ctypes.c_uint, vp]
    T.qgemv_ex.argtypes = [i32, vp, vp, vp, i32, i32, i32, ctypes.c_uint, vp]
    T.qgemv_trace_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_size_t, ctypes.POINTER(ctypes.c_int)]
    nl, nc, nf = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert T.qgemv_trace_info(ctypes.byref(nl), ctypes.byref(nc), ctypes.byref(nf)) == 0
    fmt, N, K = "Q4_K", 20000, 2560
    W = torch.from_numpy(gen.weights(fmt, N, K, 77)).cuda()
    x = torch.from_numpy(gen.normal_f32(K, 78)).cuda()
    xq0 = torch.empty(qg.qgemv_act_bytes(1, K), dtype=torch.uint8, device="cuda")
    xq1 = torch.empty_like(xq0)
    y0 = torch.empty(N, dtype=torch.float32, device="cuda")
    y1 = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    qg.qgemv_quantize_act(x, 1, K, xq0)
    qg.qgemv(fmt, W, xq0, y0, 1, N, K)
    torch.cuda.synchronize()
    assert T.qgemv_trace_begin() == 0
    s = torch.cuda.current_stream().cuda_stream
    assert T.qgemv_quantize_act_ex(x.data_ptr(), 1, K, xq1.data_ptr(), 1, s) == 0
    assert T.qgemv_ex(qg.FMT[fmt], W.data_ptr(), xq1.data_ptr(), y1.data_ptr(), 1, N, K, 1, s) == 0
    torch.cuda.synchronize()
    assert torch.equal(xq0, xq1) and y0.cpu().numpy().tobytes() == y1.cpu().numpy().tobytes()
    buf = np.zeros(2 * nc.value * nf.value, dtype=np.uint64)
    n = ctypes.c_int()
    assert T.qgemv_trace_read(buf.ctypes.data_as(ctypes.POINTER(ctypes.c_ulonglong)), buf.nbytes, ctypes.byref(n)) == 0
    assert n.value == 2
    rec = buf.reshape(2, nc.value, nf.value).astype(np.int64)
    for launch, kind in ((0, 2), (1, 1)):
        r = rec[launch][rec[launch][:, 7] != 0]
        assert len(r) > 0 and (r[:, 7] == kind).all()
        assert (r[:, 0] > 0).all() and (r[:, 0] <= r[:, 1]).all() and (r[:, 1] <= r[:, 2]).all()
        assert (r[:, 2] <= r[:, 3]).all()
    g = rec[1][rec[1][:, 7] != 0]
    assert (g[:, 8] >= g[:, 2]).all() and (g[:, 9] >= g[:, 8]).all() and (g[:, 6] < 1024).all()
    # the quantizer launch ends before the GEMV's consumers are released (programmatic dependency)
    q = rec[0][rec[0][:, 7] != 0]
    assert q[:, 3].max() <= g[:, 1].min()
