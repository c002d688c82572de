"""Pins for the oracle: each check ties it to something other than itself.

- binary16 / bfloat16 conversions: hand-chosen table + numpy's own binary16 type (a library routine).
- activation quantizer: hand-worked blocks (tests/golden), tie cases, error bound, range invariants.
- block decoders: an independent byte-walking decoder (tests/bitref.py), one-hot positional probes,
  closed forms for constant-code blocks.
- GEMV: exact rational arithmetic (fractions) on tiny shapes, dense brute force, linearity,
  row-stacking.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import qgemv_inputs as gen
from tests import bitref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------------------------
# scalar conversions

def test_fp16_decode_table():
    table = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0400: 2.0 ** -14, 0x0001: 2.0 ** -24,
             0x03FF: 1023 * 2.0 ** -24, 0x3555: 0.333251953125, 0x8000: -0.0, 0x0000: 0.0}
    for bits, val in table.items():
        assert oracle.fp16_to_f64(bits) == val, hex(bits)
    assert oracle.fp16_to_f64(0x7C00) == float("inf")
    assert np.isnan(oracle.fp16_to_f64(0x7E00))


def test_fp16_decode_all_patterns_match_numpy():
    pats = np.arange(65536, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_f64(int(p)) for p in pats])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(ref[~both_nan], got[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


def test_fp32_to_fp16_hand_table():
    cases = [
        (1.0, 0x3C00), (65504.0, 0x7BFF), (65519.0, 0x7BFF), (65520.0, 0x7C00), (-65520.0, 0xFC00),
        (1.0 + 2.0 ** -11, 0x3C00),          # tie between 1 and 1+2^-10 -> even (1.0)
        (1.0 + 3 * 2.0 ** -11, 0x3C02),      # tie between 1+2^-10 and 1+2^-9 -> even (0x3C02)
        (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000),  # half of the smallest subnormal ties to 0
        (1.5 * 2.0 ** -25, 0x0001), (3 * 2.0 ** -25, 0x0002),  # 1.5 units ties to 2 (even)
        (2.0 ** -14, 0x0400), (2.0 ** -14 - 2.0 ** -25, 0x0400),  # rounds up into the normal range
        (-0.0, 0x8000), (1e-30, 0x0000), (float("inf"), 0x7C00),
    ]
    for v, bits in cases:
        assert oracle.f32_to_fp16(np.float32(v)) == bits, (v, hex(oracle.f32_to_fp16(v)), hex(bits))
    assert (oracle.f32_to_fp16(np.float32("nan")) & 0x7C00) == 0x7C00


def test_fp32_to_fp16_matches_numpy_random():
    rng = np.random.default_rng(7)
    u = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # restrict exponents to a window around the binary16 range so most samples are interesting
    exp = rng.integers(100, 145, size=u.size).astype(np.uint32)
    bits = (u & np.uint32(0x807FFFFF)) | (exp << np.uint32(23))
    f = bits.view(np.float32)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_fp16(v) for v in f], dtype=np.uint16)
    assert np.array_equal(ref, got)


def test_bf16_decode():
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0xC040) == -3.0
    assert oracle.bf16_to_f64(0x0001) == 2.0 ** -133


# ---------------------------------------------------------------------------------------------------
# activation quantizer

def _golden_cases():
    with open(os.path.join(GOLDEN, "q8_1_worked_examples.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_quantizer_worked_examples(case):
    x = np.zeros(32, dtype=np.float32)
    x[:len(case["x_head"])] = case["x_head"]
    blk = oracle.quantize_act(x)[0]
    q = blk[4:].view(np.int8)
    exp_q = np.zeros(32, dtype=np.int8)
    exp_q[:len(case["q_head"])] = case["q_head"]
    assert np.array_equal(q, exp_q)
    assert int(blk[0]) | int(blk[1]) << 8 == int(case["d_bits"], 16)
    assert int(blk[2]) | int(blk[3]) << 8 == int(case["s_bits"], 16)


def _split(blk):
    d = int(blk[0]) | int(blk[1]) << 8
    s = int(blk[2]) | int(blk[3]) << 8
    return d, s, blk[4:36].view(np.int8).astype(np.int64)


def test_quantizer_properties_random():
    m, K = 3, 4096
    x = np.stack([gen.normal_f32(K, 11 + i) for i in range(m)])
    x[1] *= 1e-3
    x[2, :64] = 0.0
    xq = oracle.quantize_act(x).reshape(m, K // 32, 36)
    for i in range(m):
        for b in range(K // 32):
            xb = x[i, 32 * b:32 * b + 32]
            d, s, q = _split(xq[i, b])
            amax = np.float32(np.abs(xb).max())
            d32 = np.float32(amax / np.float32(127))  # numpy fp32 division (IEEE)
            assert d == np.float16(d32).view(np.uint16)  # binary16 by numpy's rounding
            assert np.abs(q).max() <= 127
            if amax == 0:
                assert (q == 0).all() and d == 0 and s == 0
                continue
            # the peak maps to +-127 and every value is within half a step (+ fp32 division error)
            assert np.abs(q).max() == 127
            err = np.abs(xb.astype(np.float64) - float(d32) * q)
            assert (err <= float(d32) * (0.5 + 1e-5)).all()
            assert (np.sign(q) * np.sign(xb) >= 0).all()
            exact_s = np.float32(np.float16(np.uint16(d).view(np.float16))) * np.float32(q.sum())
            assert s == np.float16(exact_s).view(np.uint16)


def test_quantizer_rows_independent():
    K = 256
    x = np.stack([gen.normal_f32(K, 1), gen.normal_f32(K, 2)])
    both = oracle.quantize_act(x)
    assert np.array_equal(both[0], oracle.quantize_act(x[0])[0])
    assert np.array_equal(both[1], oracle.quantize_act(x[1])[0])


def test_quantizer_scale_invariance_by_powers_of_two():
    # x * 2^k scales d32 by 2^k exactly, so the codes are unchanged (while d stays normal binary16)
    x = gen.normal_f32(1024, 5)
    base = oracle.quantize_act(x)
    for k in (-3, 2, 5):
        other = oracle.quantize_act(x * np.float32(2.0 ** k)).reshape(-1, 36)
        assert np.array_equal(other[:, 4:], base.reshape(-1, 36)[:, 4:])


# ---------------------------------------------------------------------------------------------------
# block decoders

def _rand_matrix(fmt, N, K, seed):
    return gen.weights(fmt, N, K, seed)


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
def test_decoder_matches_independent_bytewise_decoder(fmt):
    N, K = 5, 512
    W = _rand_matrix(fmt, N, K, 99)
    ref = bitref.dense_rows(fmt, W, N, K)
    got = oracle.dequant_rows(fmt, W, N, K)
    assert np.array_equal(ref, got)  # both are exact products of small integers and fp16 scales


def test_q4k_one_hot_code_positions():
    for e in range(256):
        q = np.zeros(256, dtype=np.int64)
        q[e] = 5
        blk = bitref.pack_q4k(1.0, 0.0, [1] * 8, [0] * 8, q)
        w = oracle.dequant_rows("Q4_K", blk, 1, 256)[0]
        exp = np.zeros(256)
        exp[e] = 5.0
        assert np.array_equal(w, exp), e


def test_q4k_scale_and_min_field_positions():
    for j in range(8):
        sc = [0] * 8
        mn = [0] * 8
        sc[j] = 37
        blk = bitref.pack_q4k(0.5, 0.0, sc, mn, np.ones(256, dtype=np.int64))
        w = oracle.dequant_rows("Q4_K", blk, 1, 256)[0]
        exp = np.zeros(256)
        exp[32 * j:32 * j + 32] = 0.5 * 37
        assert np.array_equal(w, exp), ("sc", j)
        sc[j] = 0
        mn[j] = 63
        blk = bitref.pack_q4k(0.5, 0.25, sc, mn, np.ones(256, dtype=np.int64))
        w = oracle.dequant_rows("Q4_K", blk, 1, 256)[0]
        exp = np.zeros(256)
        exp[32 * j:32 * j + 32] = -0.25 * 63
        assert np.array_equal(w, exp), ("mn", j)


def test_q4k_constant_block_closed_form():
    # all q = c, sc = a, mn = b  =>  w = d*a*c - dmin*b everywhere;
    # with xhat = dx*t constant: y = 256*(d*a*c - dmin*b)*dx*t per super-block
    d, dmin, a, b, c = 2.0 ** -10, 2.0 ** -11, 13, 7, 9
    blk = bitref.pack_q4k(d, dmin, [a] * 8, [b] * 8, np.full(256, c))
    w = oracle.dequant_rows("Q4_K", blk, 1, 256)[0]
    assert np.all(w == d * a * c - dmin * b)
    dx, t = 0.125, 3
    xq = np.concatenate([bitref.pack_q8_1(dx, 0.0, [t] * 32) for _ in range(8)])
    y = oracle.gemv("Q4_K", blk, xq, 1, 1, 256)[0, 0]
    assert y == 256 * (d * a * c - dmin * b) * dx * t


def test_q4k_zero_codes_and_zero_scales():
    rng = np.random.default_rng(3)
    mn = rng.integers(0, 64, 8)
    blk = bitref.pack_q4k(0.5, 2.0 ** -9, rng.integers(0, 64, 8), mn, np.zeros(256, dtype=np.int64))
    qx = rng.integers(-127, 128, 256)
    xq = np.concatenate([bitref.pack_q8_1(0.25, 0.0, qx[32 * j:32 * j + 32]) for j in range(8)])
    y = oracle.gemv("Q4_K", blk, xq, 1, 1, 256)[0, 0]
    exp = -(2.0 ** -9) * sum(int(mn[j]) * 0.25 * int(qx[32 * j:32 * j + 32].sum()) for j in range(8))
    assert y == exp
    blk0 = bitref.pack_q4k(0.5, 0.5, [0] * 8, [0] * 8, rng.integers(0, 16, 256))
    assert oracle.gemv("Q4_K", blk0, xq, 1, 1, 256)[0, 0] == 0.0


def test_q5k_one_hot_code_positions_low_and_high_bits():
    # code 5 (low bits only) and code 21 (high bit set) at every position land on that element alone
    for c in (5, 21):
        for e in range(256):
            q = np.zeros(256, dtype=np.int64)
            q[e] = c
            blk = bitref.pack_q5k(1.0, 0.0, [1] * 8, [0] * 8, q)
            w = oracle.dequant_rows("Q5_K", blk, 1, 256)[0]
            exp = np.zeros(256)
            exp[e] = float(c)
            assert np.array_equal(w, exp), (c, e)


def test_q5k_constant_block_closed_form_and_q4k_agreement():
    # all q = c, sc = a, mn = b  =>  y = 256*(d*a*c - dmin*b)*dx*t per super-block; with every high bit
    # clear, a Q5_K block decodes exactly like the Q4_K block with the same header and nibbles
    d, dmin, a, b, c = 2.0 ** -10, 2.0 ** -11, 13, 7, 25
    blk = bitref.pack_q5k(d, dmin, [a] * 8, [b] * 8, np.full(256, c))
    w = oracle.dequant_rows("Q5_K", blk, 1, 256)[0]
    assert np.all(w == d * a * c - dmin * b)
    dx, t = 0.125, 3
    xq = np.concatenate([bitref.pack_q8_1(dx, 0.0, [t] * 32) for _ in range(8)])
    assert oracle.gemv("Q5_K", blk, xq, 1, 1, 256)[0, 0] == 256 * (d * a * c - dmin * b) * dx * t
    rng = np.random.default_rng(8)
    sc, mn, q = rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 16, 256)
    b5 = bitref.pack_q5k(0.5, 0.25, sc, mn, q)
    b4 = bitref.pack_q4k(0.5, 0.25, sc, mn, q)
    assert np.array_equal(oracle.dequant_rows("Q5_K", b5, 1, 256), oracle.dequant_rows("Q4_K", b4, 1, 256))


def test_q6k_one_hot_code_positions():
    for e in range(256):
        for val in (33, 32 + 16, 32 + 31, 0):  # exercises low bits, bit 4, bit 5, the -32 floor
            q = np.full(256, 32, dtype=np.int64)
            q[e] = val
            blk = bitref.pack_q6k(1.0, [1] * 16, q)
            w = oracle.dequant_rows("Q6_K", blk, 1, 256)[0]
            exp = np.zeros(256)
            exp[e] = val - 32
            assert np.array_equal(w, exp), (e, val)


def test_q6k_bias_zero_and_single_subblock_hand_sum():
    rng = np.random.default_rng(5)
    sc = rng.integers(-64, 64, 16)
    blk = bitref.pack_q6k(0.75, sc, np.full(256, 32))
    qx = rng.integers(-127, 128, 256)
    xq = np.concatenate([bitref.pack_q8_1(0.5, 0.0, qx[32 * j:32 * j + 32]) for j in range(8)])
    assert oracle.gemv("Q6_K", blk, xq, 1, 1, 256)[0, 0] == 0.0  # q == 32 -> w == 0 exactly
    # one non-zero sub-block (index 11): y = d * sc11 * sum_{e in sub-block} (q_e - 32) * dx * qx_e
    q = np.full(256, 32, dtype=np.int64)
    q[176:192] = rng.integers(0, 64, 16)
    blk = bitref.pack_q6k(0.75, sc, q)
    y = oracle.gemv("Q6_K", blk, xq, 1, 1, 256)[0, 0]
    exp = 0.75 * int(sc[11]) * sum((int(q[e]) - 32) * 0.5 * int(qx[e]) for e in range(176, 192))
    assert y == exp


def test_q6k_bias_identity_integer():
    # sum (v-32)*x == sum v*x - 32*sum x, in integers, for any block
    rng = np.random.default_rng(8)
    v = rng.integers(0, 64, 16)
    x = rng.integers(-127, 128, 16)
    assert int(((v - 32) * x).sum()) == int((v * x).sum()) - 32 * int(x.sum())


def test_q80_one_hot_is_gather_and_accepts_minus_128():
    K = 64
    rng = np.random.default_rng(9)
    qx = rng.integers(-127, 128, K)
    xq = np.concatenate([bitref.pack_q8_1(2.0 ** -5, 0.0, qx[32 * j:32 * j + 32]) for j in range(2)])
    for k in (0, 1, 31, 32, 63):
        q = np.zeros(K, dtype=np.int64)
        q[k] = -128
        W = np.concatenate([bitref.pack_q80(0.5, q[0:32]), bitref.pack_q80(0.5, q[32:64])])
        y = oracle.gemv("Q8_0", W, xq, 1, 1, K)[0, 0]
        assert y == 0.5 * -128 * 2.0 ** -5 * int(qx[k])


def test_w8a16_integer_valued_activations_exact():
    K, N = 64, 3
    W = _rand_matrix("Q8_0", N, K, 4)
    xi = np.arange(-32, 32, dtype=np.float32)  # bf16 holds these exactly
    xb = (xi.view(np.uint32) >> 16).astype(np.uint16)
    y = oracle.w8a16(W, xb, 1, N, K)[0]
    dense = bitref.dense_rows("Q8_0", W, N, K)
    exact = [sum(Fraction(float(dense[n, k])) * int(xi[k]) for k in range(K)) for n in range(N)]
    assert all(Fraction(float(y[n])) == exact[n] for n in range(N))


# ---------------------------------------------------------------------------------------------------
# GEMV

def _exact_gemv(Wd, Xd):
    m, K = Xd.shape
    N = Wd.shape[0]
    out = np.empty((m, N), dtype=object)
    Wf = [[Fraction(float(v)) for v in row] for row in Wd]
    Xf = [[Fraction(float(v)) for v in row] for row in Xd]
    for i in range(m):
        for n in range(N):
            out[i, n] = sum(a * b for a, b in zip(Wf[n], Xf[i]))
    return out


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
def test_gemv_matches_exact_rational(fmt):
    m, N, K = 2, 3, 256
    W = _rand_matrix(fmt, N, K, 21)
    x = np.stack([gen.normal_f32(K, 31), gen.normal_f32(K, 32)])
    xq = oracle.quantize_act(x)
    y = oracle.gemv(fmt, W, xq, m, N, K)
    exact = _exact_gemv(bitref.dense_rows(fmt, W, N, K), bitref.dense_act(xq, m, K))
    for i in range(m):
        for n in range(N):
            e = float(exact[i, n])
            assert abs(y[i, n] - e) <= 1e-14 * max(1.0, abs(e)), (i, n)


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (129, 256)])
def test_gemv_matches_dense_brute_force(fmt, N, K):
    m = 2
    W = _rand_matrix(fmt, N, K, 1000 + N + K)
    x = np.stack([gen.normal_f32(K, 41), gen.normal_f32(K, 42)])
    xq = oracle.quantize_act(x)
    y = oracle.gemv(fmt, W, xq, m, N, K)
    ref = bitref.dense_act(xq, m, K) @ bitref.dense_rows(fmt, W, N, K).T
    scale = np.abs(bitref.dense_act(xq, m, K)) @ np.abs(bitref.dense_rows(fmt, W, N, K)).T
    assert (np.abs(y - ref) <= 1e-13 * scale + 1e-300).all()


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
def test_gemv_linear_in_weight_scales(fmt):
    N, K = 4, 256
    W = _rand_matrix(fmt, N, K, 5)
    xq = oracle.quantize_act(gen.normal_f32(K, 6))
    y1 = oracle.gemv(fmt, W, xq, 1, N, K)
    W2 = W.copy().reshape(N * (K // (256 if fmt != "Q8_0" else 32)), -1)
    offs = {"Q4_K": (0, 2), "Q5_K": (0, 2), "Q6_K": (208,), "Q8_0": (0,)}[fmt]
    for o in offs:  # double every fp16 scale (exponent + 1: exact for normal values)
        h = W2[:, o:o + 2].copy().view("<u2")
        W2[:, o:o + 2] = (h + np.uint16(0x0400)).view(np.uint8)
    y2 = oracle.gemv(fmt, W2.reshape(-1), xq, 1, N, K)
    assert np.array_equal(y2, 2 * y1)


@pytest.mark.parametrize("fmt", ["Q4_K", "Q5_K", "Q6_K", "Q8_0"])
def test_gemv_row_stacking_and_row_sampling(fmt):
    K = 512
    A = _rand_matrix(fmt, 3, K, 51)
    B = _rand_matrix(fmt, 5, K, 52)
    xq = oracle.quantize_act(np.stack([gen.normal_f32(K, 53), gen.normal_f32(K, 54)]))
    ya = oracle.gemv(fmt, A, xq, 2, 3, K)
    yb = oracle.gemv(fmt, B, xq, 2, 5, K)
    yab = oracle.gemv(fmt, np.concatenate([A, B]), xq, 2, 8, K)
    assert np.array_equal(yab, np.concatenate([ya, yb], axis=1))
    ys = oracle.gemv(fmt, np.concatenate([A, B]), xq, 2, 8, K, rows=[7, 0, 4])
    assert np.array_equal(ys, yab[:, [7, 0, 4]])


def test_widening_of_16_bit_activations():
    # both 16-bit kinds are subsets of binary32: widening is exact and numpy's own binary16 agrees
    h = np.array([0x3C00, 0x0001, 0x7BFF, 0x8400, 0x3555, 0x0000, 0x8000], dtype=np.uint16)
    assert np.array_equal(oracle.widen16("f16", h), h.view(np.float16).astype(np.float32))
    b = np.array([0x3F80, 0xC040, 0x0001, 0x7F7F, 0x3EAB], dtype=np.uint16)
    assert np.array_equal(oracle.widen16("bf16", b), (b.astype(np.uint32) << 16).view(np.float32))
    # the 16-bit quantizer is the fp32 one on the widened rows
    x = gen.normal_bf16(256, 5)[None, :]
    assert np.array_equal(oracle.quantize_act16("bf16", x),
                          oracle.quantize_act((x.astype(np.uint32) << 16).view(np.float32)))


# ------------------------------------------------------------------------------------------------------
# per-channel INT8 W8A16

def test_w8a16_channel_one_hot_and_scale():
    K, N = 64, 3
    x = gen.normal_bf16(K, 77)[None, :]
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    W = np.zeros((N, K), dtype=np.int8)
    W[0, 5], W[1, 63], W[2, 0] = 97, -128, 1
    sc = np.array([0.5, 2.0 ** -7, 3.0], dtype=np.float32)
    y = oracle.w8a16_channel(W, sc, x, 1, N, K)[0]
    assert y[0] == 0.5 * 97 * xv[0, 5] and y[1] == 2.0 ** -7 * -128 * xv[0, 63] and y[2] == 3.0 * xv[0, 0]


def test_w8a16_channel_integer_activations_exact_and_linear_in_scale():
    rng = np.random.default_rng(4)
    m, N, K = 2, 9, 256
    W, sc = gen.channel_weights(N, K, 9)
    xi = rng.integers(-100, 101, size=(m, K))
    xb = (xi.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # |x| <= 100: exact in bf16
    assert np.array_equal((xb.astype(np.uint32) << 16).view(np.float32), xi.astype(np.float32))
    exact = (xi @ W.reshape(N, K).astype(np.int64).T).astype(np.float64) * sc.astype(np.float64)
    y = oracle.w8a16_channel(W, sc, xb, m, N, K)
    assert np.array_equal(y, exact)
    assert np.array_equal(oracle.w8a16_channel(W, 2 * sc, xb, m, N, K), 2 * y)
    ys = oracle.w8a16_channel(W, sc, xb, m, N, K, rows=[8, 0, 3])
    assert np.array_equal(ys, y[:, [8, 0, 3]])
