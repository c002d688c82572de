"""C-ABI boundary checks that need no GPU: the library loads, exports every entry point the header
declares, sizes are right, and bad arguments are rejected on the host before anything is launched."""
import ctypes
import glob
import os
import re

import pytest

import quantized_weight_gemv_quantize_gb300 as qg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# Tests that pass fake device addresses with otherwise valid arguments run only where no GPU exists.
HAS_GPU_NODE = bool(glob.glob("/dev/nvidia[0-9]*")) or os.path.exists("/dev/nvidiactl")


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(qgemv\w*)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    qg.build()
    return qg.lib()


def test_header_declares_the_three_entry_points():
    names = _declared_functions()
    for n in ("qgemv_quantize_act", "qgemv", "qgemv_w8a16"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n  # ctypes raises AttributeError for a missing export


def test_sizes():
    assert qg.qgemv_weight_bytes("Q4_K", 256, 1024) == 147456
    assert qg.qgemv_weight_bytes("Q6_K", 1024, 3072) == 1024 * 12 * 210
    assert qg.qgemv_weight_bytes("Q8_0", 151936, 1024) == 165306368
    assert qg.qgemv_weight_bytes("Q4_K", 1, 300) == 0  # K not a block multiple
    assert qg.qgemv_weight_bytes(9, 1, 256) == 0
    assert qg.qgemv_act_bytes(1, 1024) == 1152
    assert qg.qgemv_act_bytes(8, 9728) == 8 * 304 * 36
    assert qg.qgemv_act_bytes(1, 48) == 0


def test_max_k_covers_the_workload_shapes():
    for m in range(1, 9):
        assert qg.qgemv_max_k("Q4_K", m) >= 9728
        assert qg.qgemv_max_k("Q6_K", m) >= 9728
        assert qg.qgemv_max_k("Q8_0", m) >= 16384 or m > 6
    assert qg.qgemv_max_k_w8a16(1) >= 16384
    assert qg.qgemv_max_k("Q4_K", 0) == 0 and qg.qgemv_max_k("Q4_K", 17) == 0
    # m = 9..16: one 16-row launch, or two launches of 8 and m - 8 rows for longer rows, so every K the
    # 8-row build serves is served
    for m in range(9, 17):
        for f in ("Q4_K", "Q5_K", "Q6_K", "Q8_0"):
            assert qg.qgemv_max_k(f, m) == qg.qgemv_max_k(f, 8)
        assert qg.qgemv_max_k_w8a16(m) == qg.qgemv_max_k_w8a16(8)


def test_status_strings(L):
    for s, name in qg.STATUS.items():
        assert qg.qgemv_status_string(s) == name
    assert qg.qgemv_status_string(99) == "QGEMV_ERR_UNKNOWN"


A = 0x10000  # a 16-byte aligned fake address; validation never dereferences it
B = 0x20000000
C = 0x40000000
D = 0x60000000


@pytest.mark.parametrize("args,status", [
    ((A, 0, 1024, B), 1),      # m < 1
    ((A, 17, 1024, B), 2),     # m > 16: unsupported, never a partial result
    ((A, 1, 1000, B), 1),      # K % 32
    ((A, 1, 0, B), 1),
    ((None, 1, 1024, B), 1),   # null
    ((A + 4, 1, 1024, B), 3),  # x misaligned
    ((A, 1, 1024, B + 8), 3),  # xq misaligned
    ((A, 1, 1024, A + 1024), 6),  # xq overlaps x
])
def test_quantize_rejects_on_host(L, args, status):
    x, m, K, xq = args
    assert L.qgemv_quantize_act(x, m, K, xq, None) == status


@pytest.mark.parametrize("args,status", [
    ((9, A, 1, 1024, B), 1),         # unknown input kind
    ((0, A, 1, 1024, B), 1),         # q8_1 is not an input of the quantizer
    ((2, A, 0, 1024, B), 1),         # m < 1
    ((3, A, 17, 1024, B), 2),        # m > 16
    ((2, A, 1, 1000, B), 1),         # K % 32
    ((3, A + 8, 1, 1024, B), 3),     # x misaligned (16-bit rows still need 16-byte alignment)
    ((2, A, 1, 1024, A + 1024), 6),  # xq overlaps the 2 KB of bf16 input
    ((3, A, 1, 1024, A + 2048), 0),  # adjacent, not overlapping: passes the host checks
])
def test_typed_quantize_rejects_on_host(L, args, status):
    kind, x, m, K, xq = args
    if status == 0 and HAS_GPU_NODE:
        pytest.skip("a valid call with fake addresses must never reach a GPU")
    st = L.qgemv_quantize_act_typed(kind, x, m, K, xq, 0, None)
    if status == 0:
        assert st == 4  # passes every host check, then finds no CUDA device
    else:
        assert st == status


@pytest.mark.parametrize("args,status", [
    ((7, A, B, C, 1, 16, 256), 1),         # bad format
    ((1, A, B, C, 1, 16, 300), 1),         # Q4_K needs K % 256
    ((2, A, B, C, 1, 16, 288), 1),         # Q6_K needs K % 256
    ((3, A, B, C, 1, 16, 48), 1),          # Q8_0 needs K % 32
    ((1, A, B, C, 0, 16, 256), 1),
    ((1, A, B, C, 17, 16, 256), 2),
    ((1, A, B, C, 1, 0, 256), 1),
    ((1, None, B, C, 1, 16, 256), 1),
    ((1, A + 8, B, C, 1, 16, 256), 3),     # W misaligned
    ((1, A, B + 4, C, 1, 16, 256), 3),     # xq misaligned
    ((1, A, B, C + 2, 1, 16, 256), 3),     # y misaligned
    ((1, A, B, A + 64, 1, 16, 256), 6),    # y overlaps W
    ((1, A, B, B, 1, 16, 256), 6),         # y overlaps xq
    ((1, A, B, C, 1, 16, 1 << 22), 2),     # K beyond the staging limit
])
def test_qgemv_rejects_on_host(L, args, status):
    fmt, W, xq, y, m, N, K = args
    assert L.qgemv(fmt, W, xq, y, m, N, K, None) == status


@pytest.mark.parametrize("args,status", [
    ((A, B, C, 1, 16, 48), 1),
    ((A, B, C, 17, 16, 64), 2),
    ((A, B + 2, C, 1, 16, 64), 3),
    ((A, B, B, 1, 16, 64), 6),
    ((A, B, C, 8, 16, 1 << 20), 2),
])
def test_w8a16_rejects_on_host(L, args, status):
    W, x, y, m, N, K = args
    assert L.qgemv_w8a16(W, x, y, m, N, K, None) == status


@pytest.mark.parametrize("args,status", [
    ((A, B, C, D, 0, 16, 256), 1),         # m < 1
    ((A, B, C, D, 17, 16, 256), 2),        # m > 16
    ((A, B, C, D, 1, 16, 48), 1),          # K % 32
    ((A, None, C, D, 1, 16, 256), 1),      # no scales
    ((A + 8, B, C, D, 1, 16, 256), 3),     # int8 weights misaligned
    ((A, B + 2, C, D, 1, 16, 256), 3),     # scales misaligned
    ((A, B, C, D + 2, 1, 16, 256), 3),     # y misaligned
    ((A, B, C, A, 1, 16, 256), 6),         # y overlaps the weights
    ((A, B, C, B, 1, 16, 256), 6),         # y overlaps the scales
])
def test_w8a16_channel_rejects_on_host(L, args, status):
    W, sc, x, y, m, N, K = args
    assert L.qgemv_w8a16_channel_ex(W, sc, x, y, m, N, K, 0, None) == status


SA = qg.qgemv_argmax_scratch_bytes(1)


@pytest.mark.parametrize("args,status", [
    ((4, A, B, 1, 16, 256, C, SA, D, D + 64), 1),       # W8A16 has no fused-argmax build
    ((1, A, B, 0, 16, 256, C, SA, D, D + 64), 1),       # m < 1
    ((1, A, B, 2, 16, 256, C, SA, D, D + 64), 2),       # single-row build only
    ((1, A, B, 1, 0, 256, C, SA, D, D + 64), 1),        # N < 1
    ((1, A, B, 1, 16, 200, C, SA, D, D + 64), 1),       # K % 256 for Q4_K
    ((1, A, B, 1, 16, 256, None, SA, D, D + 64), 1),    # no scratch
    ((1, A, B, 1, 16, 256, C, SA - 1, D, D + 64), 1),   # scratch too small
    ((1, A, B, 1, 16, 256, C + 8, SA, D, D + 64), 3),   # scratch misaligned
    ((1, A, B, 1, 16, 256, C, SA, D + 2, D + 64), 3),   # idx misaligned
    ((1, A, B + 4, 1, 16, 256, C, SA, D, D + 64), 3),   # activation misaligned
    ((1, A, B, 1, 16, 256, C, SA, C + 64, D + 64), 6),  # idx inside the scratch
    ((1, A, B, 1, 16, 256, C, SA, D, A + 16), 6),       # val inside the weights
    ((1, A, B, 1, 16, 256, A, SA, D, D + 64), 6),       # scratch over the weights
    ((1, A, B, 1, 16, 256, C, SA, D, D), 6),            # idx and val share memory
])
def test_argmax_rejects_on_host(L, args, status):
    fmt, W, xq, m, N, K, sc, nb, idx, val = args
    assert L.qgemv_argmax(fmt, W, xq, m, N, K, sc, nb, idx, val, 0, None) == status


def test_argmax_scratch_size(L):
    assert qg.qgemv_argmax_scratch_bytes(0) == 0 and qg.qgemv_argmax_scratch_bytes(9) == 0
    # a header line plus one (value, index) pair per CTA of the largest grid, for each activation row
    sizes = [qg.qgemv_argmax_scratch_bytes(m) for m in range(1, 9)]
    assert all(b - a == sizes[0] - 256 for a, b in zip(sizes, sizes[1:]))
    assert sizes[0] % 16 == 0 and sizes[0] >= 256 + 152 * 8


def test_failure_injection_hook(L):
    qg.qgemv_debug_fail_next(4, 2)
    assert L.qgemv_quantize_act(A, 1, 1024, B, None) == 4
    assert L.qgemv(1, A, B, C, 1, 16, 256, None) == 4
    qg.qgemv_debug_fail_next(0, 0)
    # disarmed: back to ordinary validation
    assert L.qgemv(1, A, B, C, 0, 16, 256, None) == 1


def test_python_binding_raises_with_status():
    with pytest.raises(qg.QgemvError) as ei:
        qg.qgemv("Q4_K", A, B, C, 17, 16, 256, stream=0)
    assert ei.value.status == 2


def test_route_counters_shape(L):
    qg.qgemv_route_reset()
    c = qg.qgemv_route_counts()
    assert len(c) == qg.NUM_ROUTES and all(v == 0 for v in c)


@pytest.mark.parametrize("flags", [4, 8, 0x80000000, qg.QGEMV_FLAG_PDL | qg.QGEMV_FLAG_PDL_LATE_TRIGGER | 4])
def test_quantize_rejects_unknown_flags_on_host(L, flags):
    assert L.qgemv_quantize_act_ex(A, 1, 1024, B, flags, None) == 1
    assert L.qgemv_quantize_act_typed(2, A, 1, 1024, B, flags, None) == 1


@pytest.mark.parametrize("flags", [qg.QGEMV_FLAG_PDL_LATE_TRIGGER, qg.QGEMV_FLAG_PDL | qg.QGEMV_FLAG_PDL_LATE_TRIGGER])
def test_late_trigger_is_a_quantizer_flag_only(L, flags):
    # the GEMV entry points take QGEMV_FLAG_PDL alone
    assert L.qgemv_ex(1, A, B, C, 1, 16, 256, flags, None) == 1
    assert L.qgemv_w8a16_ex(A, B, C, 1, 16, 64, flags, None) == 1


@pytest.mark.skipif(HAS_GPU_NODE, reason="checks the no-GPU path only (fake addresses must never reach a GPU)")
@pytest.mark.parametrize("flags", [qg.QGEMV_FLAG_PDL_LATE_TRIGGER, qg.QGEMV_FLAG_PDL | qg.QGEMV_FLAG_PDL_LATE_TRIGGER])
def test_quantize_accepts_the_late_trigger(L, flags):
    # passes every host check, then finds no CUDA device
    assert L.qgemv_quantize_act_ex(A, 1, 1024, B, flags, None) in (4, 5)


@pytest.mark.skipif(HAS_GPU_NODE, reason="checks the no-GPU path only (fake addresses must never reach a GPU)")
def test_valid_call_without_a_gpu_reports_cuda_error_not_a_crash(L):
    st = L.qgemv(1, A, B, C, 1, 16, 256, None)
    assert st in (4, 5)


def _mats(*triples):
    return qg.mats_array(list(triples))


@pytest.mark.parametrize("case,status", [
    (dict(fmt=1, mats=[(A, C, 16)], kind=2, act=B, xq_out=None, m=1, K=256, flags=0), 1),   # bf16 needs W8A16
    (dict(fmt=4, mats=[(A, C, 16)], kind=0, act=B, xq_out=None, m=1, K=256, flags=0), 1),   # W8A16 needs bf16
    (dict(fmt=1, mats=[(A, C, 16)], kind=0, act=B, xq_out=B + 4096, m=1, K=256, flags=0), 1),  # xq_out needs f32
    (dict(fmt=1, mats=[(A, C, 16)], kind=1, act=B + 4, xq_out=None, m=1, K=256, flags=0), 3),
    (dict(fmt=1, mats=[(A, C, 16)], kind=1, act=B, xq_out=C + 8, m=1, K=256, flags=0), 3),
    (dict(fmt=1, mats=[(A, C, 16), (A + 4096, C + 32, 16)], kind=0, act=B, xq_out=None, m=1, K=256, flags=0), 6),
    (dict(fmt=1, mats=[(A, C, 16)], kind=0, act=B, xq_out=None, m=1, K=256, flags=2), 1),   # a quantizer-only flag
    (dict(fmt=1, mats=[(A, C, 16)] * 9, kind=0, act=B, xq_out=None, m=1, K=256, flags=0), 1),  # > MAX_GROUP
    (dict(fmt=1, mats=[(A, C, 0)], kind=0, act=B, xq_out=None, m=1, K=256, flags=0), 1),
    (dict(fmt=1, mats=[(A, C, 16)], kind=0, act=B, xq_out=None, m=17, K=256, flags=0), 2),
])
def test_multi_rejects_on_host(L, case, status):
    arr = qg.mats_array(case["mats"])
    st = L.qgemv_multi(case["fmt"], len(arr), arr, case["kind"], case["act"], case["xq_out"], case["m"], case["K"],
                       case["flags"], None)
    assert st == status


@pytest.mark.skipif(HAS_GPU_NODE, reason="checks the no-GPU path only (fake addresses must never reach a GPU)")
def test_multi_valid_arguments_without_a_gpu_report_cuda_error(L):
    arr = qg.mats_array([(A, C, 16)])
    assert L.qgemv_multi(1, 1, arr, 0, B, None, 1, 256, 0, None) in (4, 5)


def test_argument_checks_are_cheap_on_the_host():
    # the per-call validation (staging limit included) must not cost more than a few microseconds
    import time
    qg.qgemv_max_k("Q8_0", 1)
    t0 = time.perf_counter()
    for _ in range(2000):
        qg.qgemv_max_k("Q8_0", 1)
        qg.qgemv_max_k_w8a16(8)
    per_call = (time.perf_counter() - t0) / 4000
    assert per_call < 20e-6, per_call



@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0", "W8A16", "W8A16_CHANNEL"])
@pytest.mark.parametrize("m", [1, 2, 8, 9, 16])
def test_k_chunk_widths(fmt, m):
    # one pass where the rows fit the staging, else as few chunks (multiples of 256 values) as fit one
    # chunk launch; beyond the served K limit, or K not a block multiple: 0
    blk = 32 if fmt in ("Q8_0", "W8A16", "W8A16_CHANNEL") else 256
    assert qg.qgemv_chunk_k(fmt, m, 2560) == 2560
    assert qg.qgemv_chunk_k(fmt, m, 131072 + blk) == 0 and qg.qgemv_chunk_k(fmt, m, blk + 1) == 0
    # widest chunk one launch can stage (a block multiple), found by search over the plan of a chunk launch
    def fits(kc):
        try:
            qg.qgemv_plan_info_chunk(fmt, m, 7, kc)
            return True
        except qg.QgemvError as e:
            assert e.status == 2
            return False
    lo, hi = 1, 131072 // blk
    while lo < hi:
        mid = (lo + hi + 1) // 2
        lo, hi = (mid, hi) if fits(mid * blk) else (lo, mid - 1)
    widest = lo * blk
    # the chunk cap: the widest chunk, or half of it for bf16 activations (room for a deeper weight ring)
    cap = (widest // (2 if fmt in ("W8A16", "W8A16_CHANNEL") else 1)) // 256 * 256
    for K in (16384, 24576, 49152, 131072):
        kc = qg.qgemv_chunk_k(fmt, m, K)
        assert 0 < kc <= K
        if kc == K:
            continue
        n = -(-K // cap)                                  # as few chunks as the cap allows, balanced
        assert kc == (-(-K // n) + 255) // 256 * 256 and kc <= cap and fits(kc)


def test_fused_argmax_needs_one_pass(L):
    # rows beyond one pass of staging at m = 1 are refused by the fused argmax (it needs whole rows in one
    # launch), on the host, before the device is touched
    blk = 256
    K = 131072
    while qg.qgemv_chunk_k("Q4_K", 1, K - blk) < K - blk:
        K -= blk
    K_one = K - blk        # largest one-pass K
    assert qg.qgemv_chunk_k("Q4_K", 1, K_one) == K_one and qg.qgemv_chunk_k("Q4_K", 1, K_one + blk) < K_one + blk
    SA = qg.qgemv_argmax_scratch_bytes(1)
    assert L.qgemv_argmax(1, A, B, 1, 16, K_one + blk, C, SA, D, D + 64, 0, None) == 2
    assert L.qgemv_argmax_noalloc(1, A, B, 1, 16, K_one + blk, D, D + 64, 0, None) == 2
