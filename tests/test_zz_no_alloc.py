"""qgemv_argmax_noalloc: the fused GEMV + argmax on the library's own static scratch.

On the host (no GPU): requests beyond the static scratch, or with m outside 1..8, are rejected before the
device is touched.  On the GPU: two calls in a row give exactly what qgemv_argmax gives on a caller-owned
scratch, and the first maximum of the GEMV's own output; the second call shows that the first left the
arrival counter at zero.  This file is collected last, so it runs both alone and after every other test.
"""
import os
import re

import numpy as np
import pytest

import qgemv_inputs as gen
import quantized_weight_gemv_quantize_gb300 as qg

torch = pytest.importorskip("torch")

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qgemv.h")
A, B, C = 0x10000, 0x20000000, 0x40000000  # fake addresses: validation never dereferences them


@pytest.fixture(scope="module")
def L():
    qg.build()
    return qg.lib()


def test_static_scratch_limit_matches_header(L):
    text = open(HEADER).read()
    limit = int(re.search(r"#define QGEMV_ARGMAX_STATIC_SCRATCH_BYTES (\d+)", text).group(1))
    assert limit == qg.QGEMV_ARGMAX_STATIC_SCRATCH_BYTES
    # room for every single-row launch, not for two activation rows
    assert qg.qgemv_argmax_scratch_bytes(1) <= limit < qg.qgemv_argmax_scratch_bytes(2)


@pytest.mark.parametrize("m,status", [(0, 1), (9, 1), (2, 2), (8, 2)])
def test_rejected_before_the_device(L, m, status):
    assert L.qgemv_argmax_noalloc(1, A, B, m, 16, 256, C, C + 64, 0, None) == status


# m = 1 calls with an argument error: each returns the argument's own status, found on the host before the
# device (or its absence, on a machine without a GPU) is consulted
@pytest.mark.parametrize("args,status", [
    ((4, A, B, 1, 16, 256, C, C + 64, 0), 1),       # W8A16 has no fused-argmax build
    ((99, A, B, 1, 16, 256, C, C + 64, 0), 1),      # unknown format
    ((1, None, B, 1, 16, 256, C, C + 64, 0), 1),    # no weights
    ((1, A, None, 1, 16, 256, C, C + 64, 0), 1),    # no activation
    ((1, A, B, 1, 16, 256, None, C + 64, 0), 1),    # no idx
    ((1, A, B, 1, 16, 256, C, None, 0), 1),         # no val
    ((1, A, B, 1, 16, 200, C, C + 64, 0), 1),       # K % 256 for Q4_K
    ((1, A, B, 1, 0, 256, C, C + 64, 0), 1),        # N < 1
    ((1, A, B, 1, 16, 256, C, C + 64, 2), 1),       # unknown flag
    ((1, A, B + 4, 1, 16, 256, C, C + 64, 0), 3),   # activation misaligned
    ((1, A, B, 1, 16, 256, C + 2, C + 64, 0), 3),   # idx misaligned
    ((1, A, B, 1, 16, 256, A + 16, C + 64, 0), 6),  # idx inside the weights
    ((1, A, B, 1, 16, 256, C, C, 0), 6),            # idx and val share memory
])
def test_m1_argument_errors_rejected_before_the_device(L, args, status):
    fmt, W, xq, m, N, K, idx, val, flags = args
    assert L.qgemv_argmax_noalloc(fmt, W, xq, m, N, K, idx, val, flags, None) == status


@pytest.mark.gpu
@pytest.mark.parametrize("flags", [0, qg.QGEMV_FLAG_PDL])
@pytest.mark.parametrize("fmt,N,K", [("Q8_0", 151936, 1024), ("Q6_K", 30000, 2560), ("Q4_K", 50000, 2560)])
def test_two_calls_equal_the_caller_scratch_entry(L, fmt, N, K, flags):
    """Two calls of the static-scratch entry issued back to back on one stream (one synchronization after
    both): each equals qgemv_argmax on a caller-owned scratch and the first maximum of the GEMV's own
    output, so the first call left the shared arrival counter at zero for the second."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qg.qgemv_device_error(reset=True)
    scratch = torch.zeros(qg.qgemv_argmax_scratch_bytes(1), dtype=torch.uint8, device="cuda")
    cases = []
    for seed in (1, 2):
        W = torch.from_numpy(gen.weights(fmt, N, K, 300 + seed)).cuda()
        x = torch.from_numpy(gen.normal_f32(K, 400 + seed)).cuda()
        xq = torch.empty(qg.qgemv_act_bytes(1, K), dtype=torch.uint8, device="cuda")
        qg.qgemv_quantize_act(x, 1, K, xq)
        y = torch.empty(N, dtype=torch.float32, device="cuda")
        qg.qgemv(fmt, W, xq, y, 1, N, K)
        idx = torch.full((2,), -7, dtype=torch.int32, device="cuda")
        val = torch.full((2,), float("nan"), dtype=torch.float32, device="cuda")
        qg.qgemv_argmax(fmt, W, xq, 1, N, K, scratch, idx[0:1], val[0:1], flags)
        cases.append((W, xq, y, idx, val))
    torch.cuda.synchronize()
    for W, xq, _, idx, val in cases:  # the two static-scratch calls, back to back
        qg.qgemv_argmax_noalloc(fmt, W, xq, 1, N, K, idx[1:2], val[1:2], flags)
    torch.cuda.synchronize()
    for seed, (_, _, y, idx, val) in zip((1, 2), cases):
        i, v, yh = idx.cpu().numpy(), val.cpu().numpy(), y.cpu().numpy()
        assert i[0] == i[1] == int(np.argmax(yh)), (fmt, seed, i)
        assert v[0].tobytes() == v[1].tobytes() == yh[i[0]].tobytes()
    assert qg.qgemv_device_error() == 0
