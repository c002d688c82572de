"""GPU parity: the CUDA path (through the C ABI) against the oracle on the same seeded inputs.

Bar: activation codes and both fp16 fields bit-exact; GEMV outputs within rel-L2 <= 1e-5 (per activation
row and overall) and max-abs <= 1e-3 * ||y_ref[i, :]||_2; bit-exact where the method makes results
independent of the launch (row stacking, rows of an m-row call vs single-row calls).
"""
import json
import os

import numpy as np
import pytest

import oracle
import qgemv_inputs as gen
import quantized_weight_gemv_quantize_gb300 as qg
from qgemv_inputs.workloads import WORKLOADS
from tests import bitref

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

REL_L2 = 1e-5
MAX_ABS = 1e-3
GUARD = 64  # guard floats after every output buffer
CANARY = np.float32(np.nan)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qg.build()
    qg.lib()
    qg.qgemv_device_error(reset=True)
    yield
    assert qg.qgemv_device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def out_buf(n):
    y = torch.full((n + GUARD,), float("nan"), dtype=torch.float32, device="cuda")
    return y


def guard_ok(y, n):
    g = y[n:].cpu().numpy()
    return np.isnan(g).all()


def row_norms(fmt, W, N, K, chunk=4096):
    """||w_n||_2 of every weight row (fp64, from the oracle's decoder)."""
    out = np.empty(N)
    for r0 in range(0, N, chunk):
        rows = range(r0, min(N, r0 + chunk))
        out[r0:r0 + len(rows)] = np.linalg.norm(oracle.dequant_rows(fmt, W, N, K, rows=rows), axis=1)
    return out


def check_close(y, ref, what="", wnorm=None, xnorm=None):
    """Tolerance of the method's outputs (fp32 accumulation of exact integer block dots):
    - rel-L2 <= 1e-5 over each output row i (when it has >= 64 values) and over the whole output;
    - max-abs <= 1e-3 * ||y_ref[i, :]||_2;
    - elementwise |err[i, n]| <= 1e-5 * ||w_n||_2 * ||xhat_i||_2, which holds for any row length
      (a single output can be tiny by cancellation, where a relative test on it says nothing)."""
    y = np.asarray(y, dtype=np.float64)
    assert np.isfinite(y).all(), f"{what}: unwritten or non-finite outputs"
    err = y - ref
    m, N = ref.shape
    for i in range(m):
        nr = np.linalg.norm(ref[i])
        if N >= 64:
            assert np.linalg.norm(err[i]) <= REL_L2 * nr, (what, i, np.linalg.norm(err[i]) / nr)
        assert np.abs(err[i]).max() <= MAX_ABS * nr, (what, i)
    if m * N >= 64:
        assert np.linalg.norm(err) <= REL_L2 * np.linalg.norm(ref), what
    if wnorm is not None:
        bound = REL_L2 * np.outer(xnorm, wnorm)
        assert (np.abs(err) <= bound).all(), (what, float((np.abs(err) / bound).max()))
    else:
        assert N >= 64, f"{what}: short rows need the elementwise bound"


def activations(m, K, seed, scale=1.0):
    return np.stack([gen.normal_f32(K, seed + 7919 * i) * np.float32(scale) for i in range(m)])


def gpu_quantize(x):
    m, K = x.shape
    xd = dev(x)
    xq = torch.empty(qg.qgemv_act_bytes(m, K), dtype=torch.uint8, device="cuda")
    qg.qgemv_quantize_act(xd, m, K, xq)
    torch.cuda.synchronize()
    return xq


def gpu_gemv(fmt, Wd, xq, m, N, K):
    y = out_buf(m * N)
    qg.qgemv(fmt, Wd, xq, y, m, N, K)
    torch.cuda.synchronize()
    assert guard_ok(y, m * N), "write past the end of y"
    return y[:m * N].cpu().numpy().reshape(m, N)


# ---------------------------------------------------------------------------------------------------
# activation quantizer: bit-exact

def _special_rows(K):
    rows = []
    r = np.zeros(K, np.float32); rows.append(r)                                  # all zero
    r = np.zeros(K, np.float32); r[::32] = 127; r[1::32] = 0.5; r[2::32] = -2.5; r[3::32] = 126.5
    rows.append(r)                                                               # ties
    r = np.zeros(K, np.float32); r[5::32] = -3.0; rows.append(r)                 # one-hot, negative
    rows.append(gen.normal_f32(K, 3) * np.float32(1e-6))                         # subnormal fp16 d
    rows.append(gen.normal_f32(K, 4) * np.float32(3e-37))                        # fp32 subnormal quotients
    rows.append(gen.normal_f32(K, 5) * np.float32(1e4))                          # large
    r = np.full(K, 1.0, np.float32); r[1::2] = 0.5; rows.append(r)               # inexact d32, tie-ish
    r = np.linspace(-1, 1, K, dtype=np.float32); rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("m,K", [(1, 32), (1, 1024), (3, 2560), (8, 9728), (2, 16384), (5, 4096), (8, 32),
                                 (1, 8192), (1, 9728), (1, 16416)])  # one-warp CTAs for long single rows
def test_quantizer_bit_exact(m, K):
    x = activations(m, K, 100 + K)
    ref = oracle.quantize_act(x).reshape(-1)
    got = gpu_quantize(x).cpu().numpy()
    assert np.array_equal(got, ref)


def test_quantizer_special_rows_bit_exact():
    K = 1024
    x = _special_rows(K)
    for i0 in range(0, x.shape[0], 8):
        xs = x[i0:i0 + 8]
        assert np.array_equal(gpu_quantize(xs).cpu().numpy(), oracle.quantize_act(xs).reshape(-1))


def _near_tie_rows(K=1024):
    """Blocks whose values sit on, or within a few ulps of, the rounding boundaries (k + 1/2) * d32."""
    rng = np.random.default_rng(5)
    rows = []
    for amax in (1.0, 3.7, 1e-3, 5e4, 0.3333333):
        blocks = []
        for b in range(K // 32):
            d32 = np.float32(np.float32(amax) / np.float32(127))
            k = rng.integers(-127, 127, 31).astype(np.float32)
            centre = ((k + np.float32(0.5)) * d32).astype(np.float32)
            steps = rng.integers(-3, 4, 31)
            v = centre.copy()
            for j, st in enumerate(steps):
                for _ in range(abs(int(st))):
                    v[j] = np.nextafter(v[j], np.float32(np.inf) if st > 0 else np.float32(-np.inf), dtype=np.float32)
            v = np.clip(v, -np.float32(amax), np.float32(amax))
            blocks.append(np.concatenate([[np.float32(amax) * (1 if b % 2 else -1)], v]).astype(np.float32))
        rows.append(np.concatenate(blocks))
    return np.stack(rows)


def test_quantizer_near_rounding_boundaries_bit_exact():
    # values on and a few ulps around every half-integer quotient, so both the reciprocal fast path and
    # its fallback to the IEEE division are taken; codes and fields must equal the oracle's bit for bit
    x = _near_tie_rows()
    xq = gpu_quantize(x)
    assert np.array_equal(xq.cpu().numpy(), oracle.quantize_act(x).reshape(-1))
    # the GEMV kernels' in-kernel quantization publishes the same blocks
    m, K = x.shape
    N = 64
    W = dev(gen.weights("Q8_0", N, K, 3))
    for i in range(m):
        xq2 = torch.empty(qg.qgemv_act_bytes(1, K), dtype=torch.uint8, device="cuda")
        y = out_buf(N)
        qg.qgemv_multi("Q8_0", [(W, y, N)], "f32", dev(x[i:i + 1]), 1, K, xq_out=xq2)
        torch.cuda.synchronize()
        assert np.array_equal(xq2.cpu().numpy(), oracle.quantize_act(x[i:i + 1]).reshape(-1))


@pytest.mark.parametrize("kind", ["bf16", "f16"])
@pytest.mark.parametrize("m,K", [(1, 32), (3, 2560), (8, 9728), (2, 16384), (1, 9728)])
def test_quantizer_16_bit_inputs_bit_exact(kind, m, K):
    rows = []
    for i in range(m):
        v = gen.normal_f32(K, 70 + i) * np.float32([1.0, 3e-5, 200.0][i % 3])
        if kind == "bf16":
            rows.append((v.view(np.uint32) >> 16).astype(np.uint16))    # truncation: any bit pattern will do
        else:
            rows.append(v.astype(np.float16).view(np.uint16))            # includes fp16 subnormals for row 1
    x16 = np.stack(rows)
    xq = torch.empty(qg.qgemv_act_bytes(m, K), dtype=torch.uint8, device="cuda")
    qg.qgemv_quantize_act_typed(kind, dev(x16), m, K, xq)
    torch.cuda.synchronize()
    ref = oracle.quantize_act16(kind, x16)
    assert np.array_equal(xq.cpu().numpy(), ref.reshape(-1))
    # and the same bytes as the fp32 entry point on the widened rows
    assert np.array_equal(gpu_quantize(oracle.widen16(kind, x16)).cpu().numpy(), ref.reshape(-1))


def test_quantizer_worked_examples_on_gpu():
    with open(os.path.join(os.path.dirname(__file__), "golden", "q8_1_worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    x = np.zeros((len(cases), 32), np.float32)
    for i, c in enumerate(cases):
        x[i, :len(c["x_head"])] = c["x_head"]
    got = gpu_quantize(x).cpu().numpy().reshape(len(cases), 36)
    for i, c in enumerate(cases):
        q = np.zeros(32, np.int8)
        q[:len(c["q_head"])] = c["q_head"]
        assert np.array_equal(got[i, 4:].view(np.int8), q), c["name"]
        assert int(got[i, 0]) | int(got[i, 1]) << 8 == int(c["d_bits"], 16), c["name"]
        assert int(got[i, 2]) | int(got[i, 3]) << 8 == int(c["s_bits"], 16), c["name"]


# ---------------------------------------------------------------------------------------------------
# GEMV

SHAPES = [(1, 256), (7, 768), (129, 2560), (333, 1024), (2560, 9728), (1000, 4096)]


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("m", [1, 2, 3, 5, 8])
def test_gemv_parity(fmt, N, K, m):
    W = gen.weights(fmt, N, K, 17 * N + K)
    x = activations(m, K, 5 + m)
    xq = gpu_quantize(x)
    xq_ref = oracle.quantize_act(x)
    assert np.array_equal(xq.cpu().numpy(), xq_ref.reshape(-1))
    y = gpu_gemv(fmt, dev(W), xq, m, N, K)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    check_close(y, oracle.gemv(fmt, W, xq_ref, m, N, K), f"{fmt} N={N} K={K} m={m}", row_norms(fmt, W, N, K), xn)


@pytest.mark.parametrize("N,K", [(301, 9472), (77, 16384), (33, 24576), (5, 9728)])
@pytest.mark.parametrize("m", [1, 3, 8])
def test_q6k_multi_warp_rows(N, K, m):
    # Q6_K rows decoded by teams of two or four warps: rows of an odd block count (a 2-byte phase that
    # alternates from row to row), K-chunked rows at m = 8, and tiles with fewer rows than teams
    W = gen.weights("Q6_K", N, K, 31 * N + K + m)
    x = activations(m, K, 9 + m)
    xq_ref = oracle.quantize_act(x)
    y = gpu_gemv("Q6_K", dev(W), gpu_quantize(x), m, N, K)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    check_close(y, oracle.gemv("Q6_K", W, xq_ref, m, N, K), f"q6_k N={N} K={K} m={m}", row_norms("Q6_K", W, N, K),
                xn)


@pytest.mark.parametrize("K", [32, 96, 4128, 8224, 16384])
@pytest.mark.parametrize("m", [1, 4])
def test_q80_rows_off_16_byte_boundaries_and_partial_chunks(K, m):
    # K % 256 != 0 puts Q8_0 rows at 2-byte offsets; long rows are streamed in several copies with a
    # shorter last one
    N = 65
    W = gen.weights("Q8_0", N, K, K + m)
    x = activations(m, K, 21)
    xq = gpu_quantize(x)
    xq_ref = oracle.quantize_act(x)
    y = gpu_gemv("Q8_0", dev(W), xq, m, N, K)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    check_close(y, oracle.gemv("Q8_0", W, xq_ref, m, N, K), f"q8_0 K={K}", row_norms("Q8_0", W, N, K), xn)


@pytest.mark.parametrize("fmt,K", [("Q4_K", 2560), ("Q5_K", 2560), ("Q6_K", 2560), ("Q8_0", 2560),
                                   # Q6_K rows decoded by two-warp teams, and rows of an odd block count, whose
                                   # 2-byte phase alternates from row to row (one pass of staging at m = 8)
                                   ("Q6_K", 9728), ("Q6_K", 9472)])
def test_gemv_rows_of_an_m_call_equal_single_row_calls(fmt, K):
    N, m = 300, 8
    W = dev(gen.weights(fmt, N, K, 3))
    x = activations(m, K, 77)
    y_all = gpu_gemv(fmt, W, gpu_quantize(x), m, N, K)
    for i in range(m):
        yi = gpu_gemv(fmt, W, gpu_quantize(x[i:i + 1]), 1, N, K)
        assert np.array_equal(y_all[i], yi[0]), i


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
def test_row_stacking_is_bit_exact(fmt):
    K = 2560
    A = gen.weights(fmt, 517, K, 1)
    B = gen.weights(fmt, 1203, K, 2)
    x = activations(2, K, 9)
    xq = gpu_quantize(x)
    ya = gpu_gemv(fmt, dev(A), xq, 2, 517, K)
    yb = gpu_gemv(fmt, dev(B), xq, 2, 1203, K)
    yab = gpu_gemv(fmt, dev(np.concatenate([A, B])), xq, 2, 1720, K)
    assert np.array_equal(yab, np.concatenate([ya, yb], axis=1))


def test_special_weight_values():
    # Q8_0 codes at -128 and 127, Q6_K sub-scales over the whole int8 range, subnormal and large fp16 d
    rng = np.random.default_rng(12)
    N, K, m = 40, 512, 3
    x = activations(m, K, 31)
    xq = gpu_quantize(x)
    xq_ref = oracle.quantize_act(x)
    blocks = []
    for n in range(N):
        for b in range(K // 32):
            q = rng.integers(-128, 128, 32)
            q[rng.integers(0, 32)] = -128
            d = [2.0 ** -24, 6.1e-5, 1.0, 100.0][(n + b) % 4]
            blocks.append(bitref.pack_q80(d, q))
    W8 = np.concatenate(blocks)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    check_close(gpu_gemv("Q8_0", dev(W8), xq, m, N, K), oracle.gemv("Q8_0", W8, xq_ref, m, N, K), "q8_0 special",
                row_norms("Q8_0", W8, N, K), xn)
    blocks = []
    for n in range(N):
        for b in range(K // 256):
            blocks.append(bitref.pack_q6k([2.0 ** -20, 0.5][n % 2], rng.integers(-128, 128, 16),
                                          rng.integers(0, 64, 256)))
    W6 = np.concatenate(blocks)
    check_close(gpu_gemv("Q6_K", dev(W6), xq, m, N, K), oracle.gemv("Q6_K", W6, xq_ref, m, N, K), "q6_k special",
                row_norms("Q6_K", W6, N, K), xn)
    blocks = []
    for n in range(N):
        for b in range(K // 256):
            blocks.append(bitref.pack_q4k([2.0 ** -20, 0.5][n % 2], [1e-3, 2.0 ** -18][n % 2],
                                          rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 16, 256)))
    W4 = np.concatenate(blocks)
    check_close(gpu_gemv("Q4_K", dev(W4), xq, m, N, K), oracle.gemv("Q4_K", W4, xq_ref, m, N, K), "q4_k special",
                row_norms("Q4_K", W4, N, K), xn)
    blocks = []
    for n in range(N):
        for b in range(K // 256):
            q = rng.integers(0, 32, 256)
            q[rng.integers(0, 256, 8)] = 31          # every high bit pattern, including all-ones codes
            blocks.append(bitref.pack_q5k([2.0 ** -20, 0.5][n % 2], [1e-3, 2.0 ** -18][n % 2],
                                          rng.integers(0, 64, 8), rng.integers(0, 64, 8), q))
    W5 = np.concatenate(blocks)
    check_close(gpu_gemv("Q5_K", dev(W5), xq, m, N, K), oracle.gemv("Q5_K", W5, xq_ref, m, N, K), "q5_k special",
                row_norms("Q5_K", W5, N, K), xn)


def _workload_shapes():
    shapes = set()
    for name in ("dense-q4k-256x1024", "dense-0.6b-class", "dense-4b-class"):
        for g in WORKLOADS[name]().gemvs:
            shapes.add((g.fmt, g.N, g.K))
    return sorted(shapes)


@pytest.mark.parametrize("fmt,N,K", _workload_shapes())
def test_workload_matrix_shapes_full_oracle(fmt, N, K):
    W = gen.weights(fmt, N, K, N * 31 + K)
    x = activations(1, K, 404)
    xq = gpu_quantize(x)
    xq_ref = oracle.quantize_act(x)
    assert np.array_equal(xq.cpu().numpy(), xq_ref.reshape(-1))
    y = gpu_gemv(fmt, dev(W), xq, 1, N, K)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, 1, K), axis=1)
    check_close(y, oracle.gemv(fmt, W, xq_ref, 1, N, K), f"{fmt} {N}x{K}", row_norms(fmt, W, N, K), xn)


@pytest.mark.parametrize("m", [2, 4, 8])
def test_skinny_batch_lm_head_sampled_rows(m):
    # the largest matrix of the 4B-class sweep at m > 1: sampled rows against the oracle
    fmt, N, K = "Q6_K", 151936, 2560
    W = gen.weights(fmt, N, K, 42)
    x = activations(m, K, 500)
    xq = gpu_quantize(x)
    xq_ref = oracle.quantize_act(x)
    y = gpu_gemv(fmt, dev(W), xq, m, N, K)
    rows = np.unique(np.concatenate([np.arange(0, N, 997), [N - 1, N - 2]]))
    ref = oracle.gemv(fmt, W, xq_ref, m, N, K, rows=rows)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    wn = np.linalg.norm(oracle.dequant_rows(fmt, W, N, K, rows=rows), axis=1)
    check_close(y[:, rows], ref, f"lm_head m={m} sampled", wn, xn)


# ---------------------------------------------------------------------------------------------------
# Integer exactness: inputs on which fp32 arithmetic is exact, so the kernel must equal the oracle bit for
# bit.  All weight scales are 2^-14 and the activation scale 2^-7, so every term the kernel forms (a scale
# product times an integer block dot or code sum) is an integer multiple of u = 2^-21, and the code ranges
# keep the sum of |terms| below 2^24 u: every partial sum, in any order, is then exact in fp32.  A wrong
# nibble, bias, index or dp4a operand anywhere changes the result by at least u.

F16_2M14, F16_2M7 = 0x0400, 0x2000  # binary16 bits of 2^-14 and 2^-7


def _exact_weights(fmt, N, K, rng):
    bb, be = bitref.BLOCK[fmt]
    W = rng.integers(0, 256, size=(N * (K // be), bb), dtype=np.uint8)
    sc = np.array([F16_2M14], dtype="<u2").view(np.uint8)
    if fmt in ("Q4_K", "Q5_K"):
        W[:, 0:2] = sc
        W[:, 2:4] = sc
    elif fmt == "Q6_K":
        W[:, 208:210] = sc
    else:
        W[:, 0:2] = sc
    return W.reshape(-1)


def _exact_act(m, K, c, rng):
    blocks = np.zeros((m * K // 32, 36), dtype=np.uint8)
    blocks[:, 0:2] = np.array([F16_2M7], dtype="<u2").view(np.uint8)
    blocks[:, 4:36] = rng.integers(-c, c + 1, size=(m * K // 32, 32)).astype(np.int8).view(np.uint8)
    return blocks.reshape(-1)


# (fmt, K, code bound c, bound on sum|term|/u per element): Q4_K (63*15 + 63)*c, Q5_K (63*31 + 63)*c,
# Q6_K 128*32*c, Q8_0 128*c
EXACT_CASES = [("Q4_K", 1024, 15, 1008 * 15), ("Q5_K", 1024, 8, 2016 * 8), ("Q6_K", 1024, 3, 4096 * 3),
               ("Q8_0", 4096, 15, 128 * 15)]


@pytest.mark.parametrize("fmt,K,c,per_elem", EXACT_CASES)
@pytest.mark.parametrize("N,m", [(67, 1), (1000, 3), (5, 8)])
def test_exact_arithmetic_inputs_give_bit_exact_outputs(fmt, K, c, per_elem, N, m):
    assert K * per_elem < 2 ** 24
    rng = np.random.default_rng(N * 7 + m + K)
    W = _exact_weights(fmt, N, K, rng)
    xq = _exact_act(m, K, c, rng)
    y = gpu_gemv(fmt, dev(W), dev(xq), m, N, K)
    ref = oracle.gemv(fmt, W, xq, m, N, K)
    assert np.array_equal(y.astype(np.float64), ref), (fmt, float(np.abs(y - ref).max()))


def _extreme_weights(fmt, N, K, rng):
    """Rows of codes at the format's limits: all largest, all smallest, a random mix of the two, and the two
    alternating.  Power-of-two scales (d = dmin = 2^-14, sub-scales +-1, minimums 0 or 1) keep every product
    and partial sum an exact fp32 value."""
    lo, hi = {"Q4_K": (0, 15), "Q5_K": (0, 31), "Q6_K": (0, 63), "Q8_0": (-128, 127)}[fmt]
    be = bitref.BLOCK[fmt][1]
    d = 2.0 ** -14
    blocks = []
    for n in range(N):
        for _ in range(K // be):
            pat = n % 4
            if pat == 0:
                q = np.full(be, hi)
            elif pat == 1:
                q = np.full(be, lo)
            elif pat == 2:
                q = np.where(rng.integers(0, 2, be) == 1, hi, lo)
            else:
                q = np.where(np.arange(be) % 2 == 0, hi, lo)
            if fmt == "Q8_0":
                blocks.append(bitref.pack_q80(d, q))
            elif fmt == "Q6_K":
                blocks.append(bitref.pack_q6k(d, rng.choice([-1, 1], 16), q))
            else:
                pack = bitref.pack_q4k if fmt == "Q4_K" else bitref.pack_q5k
                blocks.append(pack(d, d, np.ones(8, dtype=int), rng.integers(0, 2, 8), q))
    return np.concatenate(blocks)


def _extreme_act(m, K, rng):
    """q8_1 rows of codes +-127 (all +127, all -127, random signs), d = 2^-7."""
    blocks = []
    for i in range(m):
        for _ in range(K // 32):
            q = [np.full(32, 127), np.full(32, -127), rng.choice([-127, 127], 32)][i % 3]
            blocks.append(bitref.pack_q8_1(2.0 ** -7, 2.0 ** -7 * int(q.sum()), q))
    return np.concatenate(blocks)


# (fmt, K, largest |integer dot| of one block or sub-block, sub-blocks per row): each row's exact sum stays
# below 2^24 units of 2^-21, so the fp32 result is exact whatever the order of summation
EXTREME_CASES = [("Q4_K", 256, 32 * 15 * 127 + 32 * 127, 8), ("Q4_K", 2048, 32 * 15 * 127 + 32 * 127, 64),
                 ("Q5_K", 256, 32 * 31 * 127 + 32 * 127, 8), ("Q5_K", 2048, 32 * 31 * 127 + 32 * 127, 64),
                 ("Q6_K", 256, 16 * 32 * 127, 16), ("Q6_K", 2048, 16 * 32 * 127, 128),
                 ("Q8_0", 256, 32 * 128 * 127, 8), ("Q8_0", 1024, 32 * 128 * 127, 32)]


@pytest.mark.parametrize("fmt,K,per_block,nblk", EXTREME_CASES)
@pytest.mark.parametrize("m", [1, 3, 8])
def test_extreme_codes_give_bit_exact_outputs(fmt, K, per_block, nblk, m):
    # every block's integer dot at its largest magnitude (both signs): the conversion of the dp4a sums to
    # fp32 must be exact over the whole range the formats reach
    assert per_block * nblk < 2 ** 24
    rng = np.random.default_rng(K + m)
    N = 12
    W = _extreme_weights(fmt, N, K, rng)
    xq = _extreme_act(m, K, rng)
    y = gpu_gemv(fmt, dev(W), dev(xq), m, N, K)
    ref = oracle.gemv(fmt, W, xq, m, N, K)
    assert np.abs(ref).max() > 2.0 ** -21 * per_block  # the largest blocks are really there
    assert np.array_equal(y.astype(np.float64), ref), (fmt, float(np.abs(y - ref).max()))


@pytest.mark.parametrize("N,m", [(67, 1), (1000, 3), (5, 8)])
def test_w8a16_exact_arithmetic_inputs_give_bit_exact_outputs(N, m):
    K, c = 1024, 15
    assert K * 128 * c < 2 ** 24
    rng = np.random.default_rng(N + 11 * m)
    W = _exact_weights("Q8_0", N, K, rng)
    # bf16 activations that are integers times 2^-7 (exact in bf16: at most 8 significant bits)
    xv = (rng.integers(-c, c + 1, size=(m, K)) * 2.0 ** -7).astype(np.float32)
    xb = (xv.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((xb.astype(np.uint32) << 16).view(np.float32), xv)
    y = out_buf(m * N)
    qg.qgemv_w8a16(dev(W), dev(xb), y, m, N, K)
    torch.cuda.synchronize()
    assert guard_ok(y, m * N)
    ref = oracle.w8a16(W, xb, m, N, K)
    got = y[:m * N].cpu().numpy().reshape(m, N).astype(np.float64)
    assert np.array_equal(got, ref), float(np.abs(got - ref).max())


# ---------------------------------------------------------------------------------------------------
# W8A16

@pytest.mark.parametrize("N,K", [(1, 32), (7, 256), (129, 2560), (2000, 7168), (300, 16384), (77, 96)])
@pytest.mark.parametrize("m", [1, 2, 8])
def test_w8a16_parity(N, K, m):
    W = gen.weights("Q8_0", N, K, 5 * N + K)
    xb = np.stack([gen.normal_bf16(K, 60 + i) for i in range(m)])
    y = out_buf(m * N)
    qg.qgemv_w8a16(dev(W), dev(xb), y, m, N, K)
    torch.cuda.synchronize()
    assert guard_ok(y, m * N)
    xn = np.linalg.norm(np.stack([[oracle.bf16_to_f64(v) for v in row] for row in xb]), axis=1)
    check_close(y[:m * N].cpu().numpy().reshape(m, N), oracle.w8a16(W, xb, m, N, K), f"w8a16 {N}x{K} m={m}",
                row_norms("Q8_0", W, N, K), xn)


def test_w8a16_full_size_sampled_rows():
    N, K = 16384, 7168
    W = gen.weights("Q8_0", N, K, 8)
    xb = gen.normal_bf16(K, 9)[None, :]
    y = out_buf(N)
    qg.qgemv_w8a16(dev(W), dev(xb), y, 1, N, K)
    torch.cuda.synchronize()
    rows = np.arange(0, N, 61)
    xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    wn = np.linalg.norm(oracle.dequant_rows("Q8_0", W, N, K, rows=rows), axis=1)
    check_close(y[:N].cpu().numpy()[None, rows], oracle.w8a16(W, xb, 1, N, K, rows=rows), "w8a16 full", wn, xn)


# ---------------------------------------------------------------------------------------------------
# per-channel INT8 W8A16

def gpu_w8c(Wq, sc, xb, m, N, K):
    y = out_buf(m * N)
    qg.qgemv_w8a16_channel(dev(Wq), dev(sc), dev(xb), y, m, N, K)
    torch.cuda.synchronize()
    assert guard_ok(y, m * N)
    return y[:m * N].cpu().numpy().reshape(m, N)


@pytest.mark.parametrize("N,K", [(1, 32), (7, 256), (129, 2560), (2000, 7168), (300, 16384), (77, 96)])
@pytest.mark.parametrize("m", [1, 2, 8])
def test_w8a16_channel_parity(N, K, m):
    Wq, sc = gen.channel_weights(N, K, 3 * N + K)
    xb = np.stack([gen.normal_bf16(K, 80 + i) for i in range(m)])
    y = gpu_w8c(Wq, sc, xb, m, N, K)
    xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    wn = np.linalg.norm(Wq.reshape(N, K).astype(np.float64), axis=1) * sc.astype(np.float64)
    check_close(y, oracle.w8a16_channel(Wq, sc, xb, m, N, K), f"w8a16 channel {N}x{K} m={m}", wn, xn)


@pytest.mark.parametrize("N,m", [(67, 1), (1000, 3), (5, 8)])
def test_w8a16_channel_exact_arithmetic_bit_exact(N, m):
    # integer bf16 activations times 2^-7 and power-of-two row scales: every partial sum is exact in fp32
    K, c = 1024, 15
    assert K * 128 * c < 2 ** 24
    rng = np.random.default_rng(N + 5 * m)
    Wq = rng.integers(-128, 128, size=N * K).astype(np.int8)
    sc = (2.0 ** rng.integers(-12, -4, size=N)).astype(np.float32)
    xv = (rng.integers(-c, c + 1, size=(m, K)) * 2.0 ** -7).astype(np.float32)
    xb = (xv.view(np.uint32) >> 16).astype(np.uint16)
    y = gpu_w8c(Wq, sc, xb, m, N, K)
    assert np.array_equal(y.astype(np.float64), oracle.w8a16_channel(Wq, sc, xb, m, N, K))


def test_w8a16_channel_full_size_sampled_rows_and_routes():
    N, K = 16384, 7168
    Wq, sc = gen.channel_weights(N, K, 17)
    xb = gen.normal_bf16(K, 18)[None, :]
    qg.qgemv_route_reset()
    y = gpu_w8c(Wq, sc, xb, 1, N, K)
    assert qg.qgemv_route_counts()[qg.ROUTE_W8A16_CHANNEL_M1] == 1
    rows = np.arange(0, N, 61)
    xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    wn = np.linalg.norm(Wq.reshape(N, K)[rows].astype(np.float64), axis=1) * sc[rows].astype(np.float64)
    check_close(y[:, rows], oracle.w8a16_channel(Wq, sc, xb, 1, N, K, rows=rows), "w8a16 channel full", wn, xn)


# ---------------------------------------------------------------------------------------------------
# the longest supported rows

@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0", "W8A16"])
@pytest.mark.parametrize("m", [1, 8])
def test_longest_supported_rows_and_one_block_more(fmt, m):
    # K at the staging limit runs and matches the oracle; one block more is refused without a write
    w8 = fmt == "W8A16"
    wfmt = "Q8_0" if w8 else fmt
    blk = 32 if wfmt == "Q8_0" else 256
    K = qg.qgemv_max_k_w8a16(m) if w8 else qg.qgemv_max_k(fmt, m)
    assert K % blk == 0 and K > 0
    N = 5
    W = gen.weights(wfmt, N, K, 909)
    y = out_buf(m * N)
    if w8:
        xb = np.stack([gen.normal_bf16(K, 910 + i) for i in range(m)])
        qg.qgemv_w8a16(dev(W), dev(xb), y, m, N, K)
        torch.cuda.synchronize()
        ref = oracle.w8a16(W, xb, m, N, K)
        xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    else:
        x = activations(m, K, 911)
        xq = gpu_quantize(x)
        qg.qgemv(fmt, dev(W), xq, y, m, N, K)
        torch.cuda.synchronize()
        xq_ref = oracle.quantize_act(x)
        ref = oracle.gemv(fmt, W, xq_ref, m, N, K)
        xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    assert guard_ok(y, m * N)
    check_close(y[:m * N].cpu().numpy().reshape(m, N), ref, f"{fmt} K={K} m={m}", row_norms(wfmt, W, N, K), xn)
    K2 = K + blk
    W2 = dev(np.zeros(qg.qgemv_weight_bytes(wfmt, N, K2), dtype=np.uint8))
    y2 = out_buf(m * N)
    with pytest.raises(qg.QgemvError) as ei:
        if w8:
            qg.qgemv_w8a16(W2, dev(np.zeros((m, K2), dtype=np.uint16)), y2, m, N, K2)
        else:
            xq2 = torch.zeros(qg.qgemv_act_bytes(m, K2), dtype=torch.uint8, device="cuda")
            qg.qgemv(fmt, W2, xq2, y2, m, N, K2)
    assert ei.value.status == 2
    torch.cuda.synchronize()
    assert torch.isnan(y2).all()


# ---------------------------------------------------------------------------------------------------
# boundary behaviour on the device

def test_rejected_call_writes_nothing():
    K, N = 256, 16
    W = dev(gen.weights("Q4_K", N, K, 1))
    xq = torch.zeros(qg.qgemv_act_bytes(17, K), dtype=torch.uint8, device="cuda")
    y = out_buf(17 * N)
    with pytest.raises(qg.QgemvError) as ei:
        qg.qgemv("Q4_K", W, xq, y, 17, N, K)
    assert ei.value.status == 2
    torch.cuda.synchronize()
    assert torch.isnan(y).all()


def test_route_counters_witness_the_kernel_that_ran():
    qg.qgemv_route_reset()
    N, K, m = 64, 512, 3
    W = dev(gen.weights("Q6_K", N, K, 2))
    xq = gpu_quantize(activations(m, K, 2))
    gpu_gemv("Q6_K", W, xq, m, N, K)
    c = qg.qgemv_route_counts()
    assert c[0] == 1                 # one quantizer launch
    assert c[1 + 8 + (m - 1)] == 1   # Q6_K at m=3
    assert sum(c) == 2
    W5 = dev(gen.weights("Q5_K", N, K, 3))
    gpu_gemv("Q5_K", W5, xq, m, N, K)
    c = qg.qgemv_route_counts()
    assert c[qg.ROUTE_Q5_K_M1 + (m - 1)] == 1 and sum(c) == 3


def test_stream_ordering_on_a_side_stream():
    N, K = 4096, 4096
    W = dev(gen.weights("Q4_K", N, K, 6))
    x = activations(1, K, 6)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xd = dev(x)
        xq = torch.empty(qg.qgemv_act_bytes(1, K), dtype=torch.uint8, device="cuda")
        y = torch.empty(N, dtype=torch.float32, device="cuda")
        qg.qgemv_quantize_act(xd, 1, K, xq, stream=s)
        qg.qgemv("Q4_K", W, xq, y, 1, N, K, stream=s)
    s.synchronize()
    Wh = gen.weights("Q4_K", N, K, 6)
    xq_ref = oracle.quantize_act(x)
    check_close(y.cpu().numpy()[None], oracle.gemv("Q4_K", Wh, xq_ref, 1, N, K), "side stream",
                row_norms("Q4_K", Wh, N, K), np.linalg.norm(oracle.dequant_act(xq_ref, 1, K), axis=1))


# ---------------------------------------------------------------------------------------------------
# grouped launches, in-kernel quantization, programmatic dependent launch

@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
@pytest.mark.parametrize("m", [1, 3])
def test_multi_group_and_fused_quantization_equal_single_calls(fmt, m):
    K = 2560
    Ns = [2048, 512, 777]
    Ws = [dev(gen.weights(fmt, N, K, 100 + N)) for N in Ns]
    x = activations(m, K, 55)
    xq = gpu_quantize(x)
    ref = [gpu_gemv(fmt, W, xq, m, N, K) for W, N in zip(Ws, Ns)]
    ys = [out_buf(m * N) for N in Ns]
    qg.qgemv_multi(fmt, [(W, y, N) for W, y, N in zip(Ws, ys, Ns)], "q8_1", xq, m, K)
    torch.cuda.synchronize()
    for y, r, N in zip(ys, ref, Ns):
        assert guard_ok(y, m * N)
        assert np.array_equal(y[:m * N].cpu().numpy().reshape(m, N), r)
    # fp32 activations quantized inside the launch, blocks published to xq_out
    xd = dev(x)
    xq2 = torch.full((qg.qgemv_act_bytes(m, K) + 64,), 0xAB, dtype=torch.uint8, device="cuda")
    ys2 = [out_buf(m * N) for N in Ns]
    qg.qgemv_multi(fmt, [(W, y, N) for W, y, N in zip(Ws, ys2, Ns)], "f32", xd, m, K, xq_out=xq2)
    torch.cuda.synchronize()
    nq = qg.qgemv_act_bytes(m, K)
    assert np.array_equal(xq2[:nq].cpu().numpy(), xq.cpu().numpy())
    assert (xq2[nq:].cpu().numpy() == 0xAB).all()
    for y, r, N in zip(ys2, ref, Ns):
        assert guard_ok(y, m * N)
        assert np.array_equal(y[:m * N].cpu().numpy().reshape(m, N), r)


@pytest.mark.parametrize("fmt,N,K", [("Q4_K", 4096, 2560), ("Q5_K", 8192, 2560), ("Q6_K", 1024, 3072), ("Q8_0", 5000, 1024),
                                     ("Q6_K", 333, 9728)])
def test_single_row_kernel_builds_agree_bit_for_bit(fmt, N, K):
    # the register-capped build (short launches) and the streaming build (long launches) run the same
    # arithmetic in the same order: the planner may pick either for a row without changing its bits
    W = dev(gen.weights(fmt, N, K, 71 + N))
    x = activations(1, K, 72)
    xq = gpu_quantize(x)
    out = {}
    try:
        for build in (1, 2):
            qg.qgemv_tune_override(kernel_build=build)
            out[build] = gpu_gemv(fmt, W, xq, 1, N, K)
            ys = out_buf(N)
            qg.qgemv_multi(fmt, [(W, ys, N)], "f32", dev(x), 1, K)
            torch.cuda.synchronize()
            assert np.array_equal(ys[:N].cpu().numpy().reshape(1, N), out[build])
    finally:
        qg.qgemv_tune_override()
    assert np.array_equal(out[1], out[2])
    xq_ref = oracle.quantize_act(x)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, 1, K), axis=1)
    check_close(out[2], oracle.gemv(fmt, W.cpu().numpy(), xq_ref, 1, N, K), f"{fmt} builds", row_norms(fmt, W.cpu().numpy(), N, K), xn)


def test_multi_w8a16_equals_single_call():
    K, Ns = 7168, [300, 129]
    Ws = [dev(gen.weights("Q8_0", N, K, 9 + N)) for N in Ns]
    xb = dev(gen.normal_bf16(K, 4)[None, :])
    ref = []
    for W, N in zip(Ws, Ns):
        y = out_buf(N)
        qg.qgemv_w8a16(W, xb, y, 1, N, K)
        ref.append(y)
    ys = [out_buf(N) for N in Ns]
    qg.qgemv_multi("W8A16", [(W, y, N) for W, y, N in zip(Ws, ys, Ns)], "bf16", xb, 1, K)
    torch.cuda.synchronize()
    for y, r, N in zip(ys, ref, Ns):
        assert guard_ok(y, N)
        assert torch.equal(y[:N], r[:N])


def _chain(flags, W1, W2, x, N1, K1, N2, qflags=None):
    """y2 = W2 . quantize(W1 . quantize(x)): every kernel consumes the previous kernel's output.  qflags: the
    quantize launches' flags (default: flags)."""
    qf = flags if qflags is None else qflags
    s = torch.cuda.Stream()
    xq1 = torch.empty(qg.qgemv_act_bytes(1, K1), dtype=torch.uint8, device="cuda")
    y1 = torch.empty(N1, dtype=torch.float32, device="cuda")
    xq2 = torch.empty(qg.qgemv_act_bytes(1, N1), dtype=torch.uint8, device="cuda")
    y2 = torch.empty(N2, dtype=torch.float32, device="cuda")
    y3 = torch.empty(N2, dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        qg.qgemv_quantize_act_ex(x, 1, K1, xq1, qf, stream=s)
        qg.qgemv_ex("Q4_K", W1, xq1, y1, 1, N1, K1, flags, stream=s)
        qg.qgemv_quantize_act_ex(y1, 1, N1, xq2, qf, stream=s)
        qg.qgemv_ex("Q6_K", W2, xq2, y2, 1, N2, N1, flags, stream=s)
        qg.qgemv_multi("Q6_K", [(W2, y3, N2)], "f32", y1, 1, N1, flags=flags, stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
            qg.qgemv_quantize_act_ex(x, 1, K1, xq1, qf, stream=s)
            qg.qgemv_ex("Q4_K", W1, xq1, y1, 1, N1, K1, flags, stream=s)
            y1.mul_(0.5)  # an ordinary (non-PDL) kernel between library calls
            qg.qgemv_quantize_act_ex(y1, 1, N1, xq2, qf, stream=s)
            qg.qgemv_ex("Q6_K", W2, xq2, y2, 1, N2, N1, flags, stream=s)
            qg.qgemv_multi("Q6_K", [(W2, y3, N2)], "f32", y1, 1, N1, flags=flags, stream=s)
        y2.zero_()
        g.replay()
    s.synchronize()
    return y1.cpu().numpy(), y2.cpu().numpy(), y3.cpu().numpy()


@pytest.mark.parametrize("late", [False, True])
@pytest.mark.parametrize("K1,N1,N2", [(4096, 2560, 3000), (1024, 1024, 512)])
def test_programmatic_dependent_launch_chain_equals_plain_chain(late, K1, N1, N2):
    # late: the quantize launches take the late-trigger hint (the next kernel starts after their own wait).
    # The first shape runs the streaming single-row build (launches of 4 MB and more), the second the
    # register-capped one, which lets the next launch start only after its own activation staging.
    W1 = dev(gen.weights("Q4_K", N1, K1, 71))
    W2 = dev(gen.weights("Q6_K", N2, N1, 72))
    x = dev(activations(1, K1, 73))
    qg.qgemv_route_reset()
    plain = _chain(0, W1, W2, x, N1, K1, N2)
    qf = qg.QGEMV_FLAG_PDL | (qg.QGEMV_FLAG_PDL_LATE_TRIGGER if late else 0)
    pdl = _chain(qg.QGEMV_FLAG_PDL, W1, W2, x, N1, K1, N2, qflags=qf)
    assert qg.qgemv_route_counts()[qg.ROUTE_PDL] > 0
    for a_, b_ in zip(plain, pdl):
        assert np.array_equal(a_, b_)
    assert np.array_equal(plain[1], plain[2])  # in-kernel quantization == quantize + GEMV
    # and the chain is right: oracle on the same steps
    y1 = oracle.gemv("Q4_K", gen.weights("Q4_K", N1, K1, 71), oracle.quantize_act(x.cpu().numpy()), 1, N1, K1)
    assert np.linalg.norm(plain[0] - 0.5 * y1[0]) <= 1e-5 * np.linalg.norm(0.5 * y1[0])


# ---------------------------------------------------------------------------------------------------
# fused GEMV + argmax (the greedy lm_head): the chosen row equals the first maximum of the GEMV's own
# output (same per-row arithmetic, ties to the lower index), and the oracle agrees within the GEMV tolerance.

AM_FILL = -7


def gpu_argmax(fmt, Wd, xq, N, K, scratch=None, flags=0):
    if scratch is None:
        scratch = torch.zeros(qg.qgemv_argmax_scratch_bytes(1), dtype=torch.uint8, device="cuda")
    idx = torch.full((1 + GUARD,), AM_FILL, dtype=torch.int32, device="cuda")
    val = out_buf(1)
    qg.qgemv_argmax(fmt, Wd, xq, 1, N, K, scratch, idx, val, flags)
    torch.cuda.synchronize()
    assert (idx[1:] == AM_FILL).all() and guard_ok(val, 1), "write past idx / val"
    assert int(scratch[:4].view(torch.int32)[0]) == 0, "arrival counter not reset"
    return int(idx[0]), np.float32(val[0].item()), scratch


def check_argmax_against_oracle(fmt, W, xq_ref, N, K, i, v, rows=None):
    """The oracle's value at the chosen row is within the elementwise GEMV bound of the oracle's maximum
    (over all rows, or over `rows`, which must hold every row that can be the maximum)."""
    rows = np.arange(N) if rows is None else np.unique(np.append(rows, i))
    ref = oracle.gemv(fmt, W, xq_ref, 1, N, K, rows=rows)[0]
    wn = np.linalg.norm(oracle.dequant_rows(fmt, W, N, K, rows=rows), axis=1)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, 1, K))
    b = REL_L2 * wn * xn
    at = int(np.searchsorted(rows, i))
    assert abs(float(v) - ref[at]) <= b[at], (fmt, N, K, "value")
    top = int(np.argmax(ref))
    assert ref[at] >= ref[top] - (b[at] + b[top]), (fmt, N, K, i, rows[top])


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
@pytest.mark.parametrize("N,K", [(1, 256), (67, 1024), (3001, 2560), (20000, 512)])
def test_argmax_equals_first_max_of_the_gemv(fmt, N, K):
    W = gen.weights(fmt, N, K, N * 13 + K)
    x = activations(1, K, 61)
    xq = gpu_quantize(x)
    Wd = dev(W)
    y = gpu_gemv(fmt, Wd, xq, 1, N, K)[0]
    i, v, _ = gpu_argmax(fmt, Wd, xq, N, K)
    assert i == int(np.argmax(y)) and v.tobytes() == y[i].tobytes()
    check_argmax_against_oracle(fmt, W, oracle.quantize_act(x), N, K, i, v)


@pytest.mark.parametrize("fmt,K", [("Q8_0", 1024), ("Q6_K", 2560), ("Q4_K", 2560)])
def test_argmax_full_vocabulary(fmt, K):
    # the lm_head shapes of the sweeps: 151936 rows
    N = 151936
    W = gen.weights(fmt, N, K, 77)
    x = activations(1, K, 62)
    xq = gpu_quantize(x)
    Wd = dev(W)
    y = gpu_gemv(fmt, Wd, xq, 1, N, K)[0]
    qg.qgemv_route_reset()
    i, v, _ = gpu_argmax(fmt, Wd, xq, N, K)
    assert qg.qgemv_route_counts()[qg.ROUTE_ARGMAX] == 1
    assert i == int(np.argmax(y)) and v.tobytes() == y[i].tobytes()
    # every row whose GEMV value is within a generous margin of the maximum (the rest cannot be the
    # oracle's maximum: the GEMV error per row is far below the margin)
    cand = np.nonzero(y >= y[i] - 1e-3 * abs(float(y[i])) - 1e-3)[0]
    assert len(cand) < 2000
    check_argmax_against_oracle(fmt, W, oracle.quantize_act(x), N, K, i, v, rows=cand)


def test_argmax_two_calls_on_one_scratch_and_pdl():
    fmt, N, K = "Q6_K", 40000, 1024
    scratch = torch.zeros(qg.qgemv_argmax_scratch_bytes(1), dtype=torch.uint8, device="cuda")
    for seed, flags in ((1, 0), (2, 0), (3, qg.QGEMV_FLAG_PDL), (4, qg.QGEMV_FLAG_PDL)):
        W = gen.weights(fmt, N, K, 500 + seed)
        xq = gpu_quantize(activations(1, K, 600 + seed))
        Wd = dev(W)
        y = gpu_gemv(fmt, Wd, xq, 1, N, K)[0]
        i, v, scratch = gpu_argmax(fmt, Wd, xq, N, K, scratch, flags)
        assert i == int(np.argmax(y)) and v.tobytes() == y[i].tobytes(), seed


@pytest.mark.parametrize("fmt", ["Q4_K", "Q6_K", "Q8_0"])
def test_argmax_ties_go_to_the_lowest_row(fmt):
    N, K = 5000, 1024
    rb = bitref.BLOCK[fmt][0] * (K // bitref.BLOCK[fmt][1])
    W = gen.weights(fmt, N, K, 909).reshape(N, rb)
    x = activations(1, K, 63)
    xq = gpu_quantize(x)
    y = gpu_gemv(fmt, dev(W), xq, 1, N, K)[0]
    r = int(np.argmax(y))
    # copies of the best row before it, in another CTA's tiles, and after it: identical bytes give
    # identical values, so the lowest copy must win
    for p in sorted({r // 3, r // 2, (r + N) // 2, N - 1} - {r}):
        W[p] = W[r]
    Wd = dev(W)
    y2 = gpu_gemv(fmt, Wd, xq, 1, N, K)[0]
    i, v, _ = gpu_argmax(fmt, Wd, xq, N, K)
    first = int(np.nonzero(y2 == y2.max())[0][0])
    assert i == first == min(r // 3, r) and v.tobytes() == y2[r].tobytes()
    # every row the same, every value negative: row 0 (an initial best of 0 or a lost -inf would fail)
    Wall = np.repeat(W[r:r + 1], N, axis=0)
    xn = -x if y[r] > 0 else x
    xqn = gpu_quantize(xn)
    yn = gpu_gemv(fmt, dev(Wall), xqn, 1, N, K)[0]
    assert (yn < 0).all() and (yn == yn[0]).all()
    i, v, _ = gpu_argmax(fmt, dev(Wall), xqn, N, K)
    assert i == 0 and v.tobytes() == yn[0].tobytes()


@pytest.mark.parametrize("fmt", ["Q4_K", "Q6_K", "Q8_0"])
def test_argmax_orders_nan_first_like_numpy(fmt):
    """A weight row whose fp16 scale is NaN gives a NaN output row; the argmax then names the first NaN
    row (numpy.argmax / torch.argmax order: NaN above every number, the lower row among NaNs)."""
    N, K = 20000, 1024
    rb = bitref.BLOCK[fmt][0] * (K // bitref.BLOCK[fmt][1])
    d_at = {"Q4_K": 0, "Q6_K": 208, "Q8_0": 0}[fmt]
    W = gen.weights(fmt, N, K, 919).reshape(N, rb)
    nan_rows = (N - 7, 9001, 12345)
    for r in nan_rows:
        W[r, d_at:d_at + 2] = np.frombuffer(np.uint16(0x7E00).tobytes(), np.uint8)
    x = activations(1, K, 64)
    xq = gpu_quantize(x)
    Wd = dev(W)
    y = out_buf(N)
    qg.qgemv(fmt, Wd, xq, y, 1, N, K)
    torch.cuda.synchronize()
    yh = y[:N].cpu().numpy()
    assert np.isnan(yh[list(nan_rows)]).all() and np.isfinite(np.delete(yh, nan_rows)).all()
    i, v, _ = gpu_argmax(fmt, Wd, xq, N, K)
    assert i == int(np.argmax(yh)) == min(nan_rows) and np.isnan(v)


# ---------------------------------------------------------------------------------------------------
# Rows longer than one pass of activation staging: one launch per K-chunk, each reading only its chunk of
# every weight row and staging only its chunk of the activation; later chunks add to y in stream order.

LONG_FMTS = ["Q4_K", "Q5_K", "Q6_K", "Q8_0", "W8A16", "W8A16_CHANNEL"]


def one_pass_limit(fmt, m):
    """Largest K (a block multiple) that still runs in one pass of staging at m rows."""
    blk = 32 if fmt in ("Q8_0", "W8A16", "W8A16_CHANNEL") else 256
    lo, hi = 1, qg.qgemv_max_k("Q8_0", m) // blk
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if qg.qgemv_chunk_k(fmt, m, mid * blk) == mid * blk:
            lo = mid
        else:
            hi = mid - 1
    return lo * blk


def gpu_any(fmt, m, N, K, seed, flags=0):
    """(y from the GPU, oracle y, weight-row norms, activation-row norms) for one call of `fmt`."""
    if fmt == "W8A16_CHANNEL":
        Wq, sc = gen.channel_weights(N, K, seed)
        xb = np.stack([gen.normal_bf16(K, seed + 1 + i) for i in range(m)])
        y = out_buf(m * N)
        qg.qgemv_w8a16_channel(dev(Wq), dev(sc), dev(xb), y, m, N, K, flags)
        ref = oracle.w8a16_channel(Wq, sc, xb, m, N, K)
        wn = np.linalg.norm(Wq.reshape(N, K).astype(np.float64), axis=1) * sc.astype(np.float64)
        xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    elif fmt == "W8A16":
        W = gen.weights("Q8_0", N, K, seed)
        xb = np.stack([gen.normal_bf16(K, seed + 1 + i) for i in range(m)])
        y = out_buf(m * N)
        qg.qgemv_w8a16_ex(dev(W), dev(xb), y, m, N, K, flags)
        ref = oracle.w8a16(W, xb, m, N, K)
        wn = row_norms("Q8_0", W, N, K)
        xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    else:
        W = gen.weights(fmt, N, K, seed)
        x = activations(m, K, seed + 1)
        xq = gpu_quantize(x)
        y = out_buf(m * N)
        qg.qgemv_ex(fmt, dev(W), xq, y, m, N, K, flags)
        xq_ref = oracle.quantize_act(x)
        ref = oracle.gemv(fmt, W, xq_ref, m, N, K)
        wn = row_norms(fmt, W, N, K)
        xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    torch.cuda.synchronize()
    assert guard_ok(y, m * N), "write past the end of y"
    return y[:m * N].cpu().numpy().reshape(m, N), ref, wn, xn


@pytest.mark.parametrize("fmt", LONG_FMTS)
@pytest.mark.parametrize("m", [2, 8, 12, 16])
def test_rows_just_beyond_one_pass_run_as_k_chunks(fmt, m):
    K = (one_pass_limit(fmt, m) // 256 + 1) * 256
    kc = qg.qgemv_chunk_k(fmt, m, K)
    assert 0 < kc < K and kc % 256 == 0
    chunks = -(-K // kc)
    qg.qgemv_route_reset()
    y, ref, wn, xn = gpu_any(fmt, m, 67, K, 1000 + m)
    routes = qg.qgemv_route_counts()
    assert routes[qg.ROUTE_CHUNKED] == chunks
    check_close(y, ref, f"{fmt} m={m} K={K} in {chunks} chunks", wn, xn)


@pytest.mark.parametrize("fmt", LONG_FMTS)
def test_many_k_chunks_with_programmatic_dependent_launch(fmt):
    m, N, K = 8, 33, 49152
    kc = qg.qgemv_chunk_k(fmt, m, K)
    assert -(-K // kc) >= 3
    y, ref, wn, xn = gpu_any(fmt, m, N, K, 2000, flags=qg.QGEMV_FLAG_PDL)
    check_close(y, ref, f"{fmt} m={m} K={K}", wn, xn)


@pytest.mark.parametrize("fmt", ["Q8_0", "W8A16", "W8A16_CHANNEL"])
def test_k_chunked_exact_arithmetic_is_bit_exact(fmt):
    # unit codes keep every partial sum exact in fp32 (K * 128 < 2^24 terms of at most 2^7 u), so each chunk
    # and the sum over chunks must equal the oracle bit for bit
    m, N, K = 8, 29, 20480
    assert qg.qgemv_chunk_k(fmt, m, K) < K and K * 128 < 2 ** 24
    rng = np.random.default_rng(77)
    y = out_buf(m * N)
    if fmt == "Q8_0":
        W = _exact_weights("Q8_0", N, K, rng)
        xq = _exact_act(m, K, 1, rng)
        qg.qgemv("Q8_0", dev(W), dev(xq), y, m, N, K)
        ref = oracle.gemv("Q8_0", W, xq, m, N, K)
    else:
        xv = (rng.integers(-1, 2, size=(m, K)) * 2.0 ** -7).astype(np.float32)
        xb = (xv.view(np.uint32) >> 16).astype(np.uint16)
        if fmt == "W8A16":
            W = _exact_weights("Q8_0", N, K, rng)
            qg.qgemv_w8a16(dev(W), dev(xb), y, m, N, K)
            ref = oracle.w8a16(W, xb, m, N, K)
        else:
            Wq = rng.integers(-128, 128, size=N * K).astype(np.int8)
            sc = (2.0 ** rng.integers(-12, -4, size=N)).astype(np.float32)
            qg.qgemv_w8a16_channel(dev(Wq), dev(sc), dev(xb), y, m, N, K)
            ref = oracle.w8a16_channel(Wq, sc, xb, m, N, K)
    torch.cuda.synchronize()
    assert guard_ok(y, m * N)
    got = y[:m * N].cpu().numpy().reshape(m, N).astype(np.float64)
    assert np.array_equal(got, ref), float(np.abs(got - ref).max())


@pytest.mark.parametrize("fmt,m", [("Q6_K", 8), ("Q4_K", 16), ("Q8_0", 12)])
def test_k_chunked_groups_and_in_launch_quantization_equal_single_calls(fmt, m):
    # two matrices in one call, fp32 activations quantized inside every chunk launch (each publishing its
    # chunk's q8_1 blocks): bit-identical to single calls on separately quantized activations
    K = (one_pass_limit(fmt, m) // 256 + 2) * 256
    assert qg.qgemv_chunk_k(fmt, m, K) < K
    Ns = (70, 45)
    Ws = [dev(gen.weights(fmt, n, K, 3000 + n)) for n in Ns]
    x = activations(m, K, 3100)
    xq = gpu_quantize(x)
    singles = [gpu_gemv(fmt, W, xq, m, n, K) for W, n in zip(Ws, Ns)]
    ys = [out_buf(m * n) for n in Ns]
    xq_out = torch.zeros(qg.qgemv_act_bytes(m, K), dtype=torch.uint8, device="cuda")
    qg.qgemv_multi(fmt, [(W, y, n) for W, y, n in zip(Ws, ys, Ns)], "f32", dev(x), m, K, xq_out=xq_out)
    torch.cuda.synchronize()
    assert torch.equal(xq_out, xq)
    for y, n, ref in zip(ys, Ns, singles):
        assert guard_ok(y, m * n)
        assert y[:m * n].cpu().numpy().reshape(m, n).tobytes() == ref.tobytes()


def test_w8a16_large_hidden_down_projection_at_m8_sampled_rows():
    # the 16384 -> 7168 projection at m = 8, beyond one pass of staging (two chunks or more)
    m, N, K = 8, 7168, 16384
    assert qg.qgemv_chunk_k("W8A16", m, K) < K
    W = gen.weights("Q8_0", N, K, 4100)
    xb = np.stack([gen.normal_bf16(K, 4101 + i) for i in range(m)])
    y = out_buf(m * N)
    qg.qgemv_w8a16(dev(W), dev(xb), y, m, N, K)
    torch.cuda.synchronize()
    assert guard_ok(y, m * N)
    rows = np.unique(np.concatenate([np.arange(0, N, 97), [N - 1]]))
    xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    wn = np.linalg.norm(oracle.dequant_rows("Q8_0", W, N, K, rows=rows), axis=1)
    got = y[:m * N].cpu().numpy().reshape(m, N)[:, rows]
    check_close(got, oracle.w8a16(W, xb, m, N, K, rows=rows), "w8a16 16384->7168 m=8", wn, xn)


# ---------------------------------------------------------------------------------------------------
# m = 9..16: the 16-row build (rows past m staged as zeros, never stored), or two launches of 8 and m - 8
# rows where K is beyond that build's activation staging

MEDIUM_SHAPES = [(7, 768), (333, 1024), (1000, 4096), (2560, 9728)]


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
@pytest.mark.parametrize("N,K", MEDIUM_SHAPES)
@pytest.mark.parametrize("m", [9, 12, 16])
def test_medium_m_parity(fmt, N, K, m):
    W = gen.weights(fmt, N, K, 19 * N + K)
    x = activations(m, K, 40 + m)
    xq = gpu_quantize(x)
    xq_ref = oracle.quantize_act(x)
    assert np.array_equal(xq.cpu().numpy(), xq_ref.reshape(-1))
    qg.qgemv_route_reset()
    y = gpu_gemv(fmt, dev(W), xq, m, N, K)
    single = qg.qgemv_plan_info(fmt, m, N, K)["kernel_build"] == 10
    c = qg.qgemv_route_counts()
    assert c[qg.ROUTE_M16] == (1 if single else 0)
    xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    check_close(y, oracle.gemv(fmt, W, xq_ref, m, N, K), f"{fmt} N={N} K={K} m={m}", row_norms(fmt, W, N, K), xn)


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
@pytest.mark.parametrize("K", [2560, 9728])
def test_medium_m_rows_equal_single_row_calls(fmt, K):
    # each output row's arithmetic does not depend on m, on the padding or on the two-launch split
    N, m = 300, 16
    W = dev(gen.weights(fmt, N, K, 5))
    x = activations(m, K, 78)
    y_all = gpu_gemv(fmt, W, gpu_quantize(x), m, N, K)
    for i in (0, 7, 8, 15):
        yi = gpu_gemv(fmt, W, gpu_quantize(x[i:i + 1]), 1, N, K)
        assert np.array_equal(y_all[i], yi[0]), i
    y13 = gpu_gemv(fmt, W, gpu_quantize(x[:13]), 13, N, K)
    assert np.array_equal(y13, y_all[:13])


@pytest.mark.parametrize("fmt,K,c,per_elem", EXACT_CASES)
def test_medium_m_exact_arithmetic_bit_exact(fmt, K, c, per_elem):
    rng = np.random.default_rng(K + 16)
    N, m = 300, 16
    W = _exact_weights(fmt, N, K, rng)
    xq = _exact_act(m, K, c, rng)
    y = gpu_gemv(fmt, dev(W), dev(xq.reshape(-1)), m, N, K)
    assert np.array_equal(y.astype(np.float64), oracle.gemv(fmt, W, xq, m, N, K)), fmt


@pytest.mark.parametrize("N,K", [(129, 2560), (300, 16384 // 4), (77, 96)])
@pytest.mark.parametrize("m", [11, 16])
def test_medium_m_w8a16_and_channel_parity(N, K, m):
    W = gen.weights("Q8_0", N, K, 3 * N + K)
    xb = np.stack([gen.normal_bf16(K, 700 + i) for i in range(m)])
    y = out_buf(m * N)
    qg.qgemv_w8a16(dev(W), dev(xb), y, m, N, K)
    torch.cuda.synchronize()
    assert guard_ok(y, m * N)
    xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    check_close(y[:m * N].cpu().numpy().reshape(m, N), oracle.w8a16(W, xb, m, N, K), f"w8a16 m={m}",
                row_norms("Q8_0", W, N, K), xn)
    Wq, sc = gen.channel_weights(N, K, 9 + m)
    y2 = gpu_w8c(Wq, sc, xb, m, N, K)
    wn = np.linalg.norm(Wq.reshape(N, K).astype(np.float64), axis=1) * sc.astype(np.float64)
    check_close(y2, oracle.w8a16_channel(Wq, sc, xb, m, N, K), f"w8c m={m}", wn, xn)


@pytest.mark.parametrize("fmt,K", [("Q4_K", 1024), ("Q6_K", 1024), ("Q8_0", 1024), ("Q6_K", 9728)])
def test_medium_m_multi_and_fused_quantization_equal_single_calls(fmt, K):
    m = 12
    Ns = (512, 300, 1024)
    Ws = [dev(gen.weights(fmt, N, K, 60 + j)) for j, N in enumerate(Ns)]
    x = activations(m, K, 61)
    xd = dev(x)
    xq = gpu_quantize(x)
    ref = [gpu_gemv(fmt, W, xq, m, N, K) for W, N in zip(Ws, Ns)]
    ys = [out_buf(m * N) for N in Ns]
    nq = qg.qgemv_act_bytes(m, K)
    xq_out = torch.full((nq + 64,), 0xAB, dtype=torch.uint8, device="cuda")
    qg.qgemv_multi(fmt, [(W, y, N) for W, y, N in zip(Ws, ys, Ns)], "f32", xd, m, K, xq_out=xq_out)
    torch.cuda.synchronize()
    assert torch.equal(xq_out[:nq], xq) and (xq_out[nq:].cpu().numpy() == 0xAB).all()
    for y, r, N in zip(ys, ref, Ns):
        assert guard_ok(y, m * N)
        assert np.array_equal(y[:m * N].cpu().numpy().reshape(m, N), r)


@pytest.mark.parametrize("fmt", ["Q4_K", "Q6_K", "Q8_0", "W8A16"])
def test_medium_m_longest_rows_and_one_block_more(fmt):
    m, N = 16, 5
    w8 = fmt == "W8A16"
    wfmt = "Q8_0" if w8 else fmt
    blk = 32 if wfmt == "Q8_0" else 256
    K = qg.qgemv_max_k_w8a16(m) if w8 else qg.qgemv_max_k(fmt, m)
    W = gen.weights(wfmt, N, K, 919)
    if w8:
        xb = np.stack([gen.normal_bf16(K, 920 + i) for i in range(m)])
        y = out_buf(m * N)
        qg.qgemv_w8a16(dev(W), dev(xb), y, m, N, K)
        torch.cuda.synchronize()
        ref = oracle.w8a16(W, xb, m, N, K)
        xn = np.linalg.norm((xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64), axis=1)
    else:
        x = activations(m, K, 921)
        xq_ref = oracle.quantize_act(x)
        y = out_buf(m * N)
        qg.qgemv(fmt, dev(W), gpu_quantize(x), y, m, N, K)
        torch.cuda.synchronize()
        ref = oracle.gemv(fmt, W, xq_ref, m, N, K)
        xn = np.linalg.norm(oracle.dequant_act(xq_ref, m, K), axis=1)
    assert guard_ok(y, m * N)
    check_close(y[:m * N].cpu().numpy().reshape(m, N), ref, f"{fmt} K={K} m=16", row_norms(wfmt, W, N, K), xn)
    K2 = K + blk
    y2 = out_buf(m * N)
    with pytest.raises(qg.QgemvError) as ei:
        W2 = dev(np.zeros(qg.qgemv_weight_bytes(wfmt, N, K2), dtype=np.uint8))
        if w8:
            qg.qgemv_w8a16(W2, dev(np.zeros((m, K2), dtype=np.uint16)), y2, m, N, K2)
        else:
            qg.qgemv(fmt, W2, torch.zeros(qg.qgemv_act_bytes(m, K2), dtype=torch.uint8, device="cuda"), y2, m, N, K2)
    assert ei.value.status == 2
    torch.cuda.synchronize()
    assert torch.isnan(y2).all()


@pytest.mark.parametrize("fmt,N,K,m", [("Q4_K", 19456 // 4, 2560, 8), ("Q4_K", 2560, 4096, 4), ("Q4_K", 777, 1024, 5),
                                       ("Q4_K", 6144, 2560, 6), ("Q4_K", 33, 2560, 7),
                                       # Q6_K pairs run in a build of their own (8 rows)
                                       ("Q6_K", 151936 // 8, 2560, 8), ("Q6_K", 1001, 4096, 8), ("Q6_K", 33, 2560, 8),
                                       ("Q6_K", 500, 1024, 8)])
def test_row_pairs_give_bit_identical_rows(fmt, N, K, m):
    # teams that decode two rows at once run each row's arithmetic unchanged: forcing pairs on and off
    # gives the same bits (and matches the oracle)
    w8 = fmt == "W8A16"
    W = dev(gen.weights("Q8_0" if w8 else fmt, N, K, 4242))
    if w8:
        xb = dev(np.stack([gen.normal_bf16(K, 4300 + i) for i in range(m)]))
    else:
        xq = gpu_quantize(activations(m, K, 4300))
    outs = []
    try:
        for mode in (1, 2):
            qg.qgemv_tune_pairs(mode)
            y = out_buf(m * N)
            if w8:
                qg.qgemv_w8a16(W, xb, y, m, N, K)
            else:
                qg.qgemv(fmt, W, xq, y, m, N, K)
            torch.cuda.synchronize()
            assert guard_ok(y, m * N)
            outs.append(y[:m * N].cpu().numpy())
    finally:
        qg.qgemv_tune_pairs(0)
    assert np.array_equal(outs[0], outs[1])
    assert np.isfinite(outs[0]).all()


@pytest.mark.parametrize("fmt,N,K,m", [("Q4_K", 19456, 2560, 1), ("Q6_K", 2560, 9728, 1), ("Q6_K", 2560, 9728, 8),
                                       ("Q8_0", 151936, 1024, 1), ("Q4_K", 19456, 2560, 8)])
def test_repeated_launches_are_bit_identical(fmt, N, K, m):
    # every row's summation order is fixed by (format, K): the multi-warp reduction, the row pairs and the
    # grid-stride tile order do not make a run-to-run difference
    W = dev(gen.weights(fmt, N, K, 31337))
    xq = gpu_quantize(activations(m, K, 31338))
    first = gpu_gemv(fmt, W, xq, m, N, K)
    for _ in range(3):
        assert np.array_equal(gpu_gemv(fmt, W, xq, m, N, K), first)


@pytest.mark.parametrize("mode", ["fused", "percall"])
def test_decode_sweep_with_programmatic_launch_equals_plain_calls(mode):
    # The 0.6B-class decode sweep as the benchmark issues it (same-input groups, fp32 activations quantized in
    # the launch or by a quantize launch, the late-trigger hint before the short down projections, the capped
    # single-row build's later trigger, one weight tile before each dependency wait), replayed as one CUDA
    # graph with programmatic dependent launch: every output equals the same calls issued without it.
    import bench
    wl = WORKLOADS["dense-0.6b-class"]()
    sw = bench.Sweep(wl, torch, qg, gen)
    stream = torch.cuda.Stream()
    sw.d_out.fill_(0xFF)
    with torch.cuda.stream(stream):
        bench.Sweep.run(sw.calls(mode, False), stream.cuda_stream)
    stream.synchronize()
    ref = sw.d_out.clone()
    sw.d_out.fill_(0xFF)
    pdl_calls = sw.calls(mode, True)
    assert any(c[2][4] & qg.QGEMV_FLAG_PDL_LATE_TRIGGER for c in pdl_calls if c[0] == "quantize")
    g = bench._graph_of(torch, pdl_calls, stream)
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    stream.synchronize()
    assert torch.equal(sw.d_out, ref)
    for i, gm in enumerate(wl.gemvs):
        y = ref[sw.youts[i]:sw.youts[i] + wl.m * gm.N * 4].view(torch.float32)
        assert torch.isfinite(y).all(), (i, gm.fmt, gm.N, gm.K)
