"""Host-side check of the GEMV kernel's index arithmetic against the launch plan (no GPU needed).

For each plan the library would launch, every tile's bulk-copy range, tail bytes and the decoders'
furthest shared-memory reads are recomputed from the kernel's formulas and checked against the ring slot,
the weight allocation and the shared-memory budget.
"""
import numpy as np
import pytest

import quantized_weight_gemv_quantize_gb300 as qg
from qgemv_inputs.workloads import WORKLOADS

SMEM_CAP = 232448
BAR_BYTES = 128  # full + empty mbarrier (8 bytes each) per ring slot, 8 slots
NC = 8           # consumer warps per CTA
# furthest byte a unit decoder reads past the start of its block (exclusive), from the kernel's loads
READ_END = {"Q4_K": 144, "Q5_K": 176, "Q6_K": 212, "Q8_0": 38, "W8A16": 38, "W8A16_CHANNEL": 32}
BLOCK = {"Q4_K": (144, 256), "Q5_K": (176, 256), "Q6_K": (210, 256), "Q8_0": (34, 32), "W8A16": (34, 32),
         "W8A16_CHANNEL": (32, 32)}


def _shapes():
    out = set()
    for name in ("dense-q4k-256x1024", "dense-0.6b-class", "dense-4b-class", "w8a16-large"):
        wl = WORKLOADS[name]()
        for g in wl.gemvs:
            out.add(("W8A16" if g.w8a16 else g.fmt, g.N, g.K))
    for fmt in ("Q4_K", "Q5_K", "Q6_K", "Q8_0", "W8A16", "W8A16_CHANNEL"):
        for N in (1, 7, 129, 333, 1000, 2560):
            for K in (256, 768, 2560, 4096, 9728):
                out.add((fmt, N, K))
    for K in (32, 96, 224, 8224):
        out.add(("Q8_0", 77, K))
        out.add(("W8A16", 77, K))
        out.add(("W8A16_CHANNEL", 77, K))
    # rows longer than one pass of staging at some m (K-chunked), ragged last chunks, the K limit
    for fmt in ("Q4_K", "Q5_K", "Q6_K", "Q8_0", "W8A16", "W8A16_CHANNEL"):
        for N, K in ((7, 131072), (129, 20480), (333, 24576), (5, 17664)):
            out.add((fmt, N, K))
    for fmt in ("Q8_0", "W8A16", "W8A16_CHANNEL"):
        out.add((fmt, 77, 16416))
        out.add((fmt, 300, 16384))
    out.add(("W8A16", 7168, 16384))
    return sorted(out)


def check_chunked_plan(fmt, m, N, K, c0, kw, p):
    """One K-chunk launch covering values [c0, c0 + kw) of every row: each tile row is its own copy of the
    aligned superset of the row's chunk bytes, at p["slot_row_stride"] in the slot."""
    bb, be = BLOCK[fmt]
    RBF = K // be * bb                 # whole weight row in global memory
    SEG = kw // be * bb                # the chunk's bytes of a row
    OFF = c0 // be * bb
    total = N * RBF
    assert p["row_bytes"] == SEG and c0 % 256 == 0
    R, S, slot, G = p["rows_per_tile"], p["stages"], p["stage_bytes"], p["team_warps"]
    stride = p["slot_row_stride"]
    assert stride % 16 == 0 and stride >= SEG + 30
    assert 1 <= R <= N and 2 <= S <= 8 and slot % 128 == 0 and slot >= R * stride
    assert BAR_BYTES + p["red_bytes"] + p["x_stage_bytes"] + S * slot == p["smem"] <= SMEM_CAP
    assert p["num_tiles"] == -(-N // R) and 1 <= p["grid"] <= p["num_tiles"]
    n = np.arange(N, dtype=np.int64)
    rr = n % R                         # row of its tile
    s = n * RBF + OFF
    e = s + SEG
    al = s & ~15
    ce = np.minimum((e + 15) & ~15, total & ~15)
    assert (al >= 0).all() and (ce >= al).all() and (ce <= total).all() and ((ce - al) % 16 == 0).all()
    assert (e - al <= stride).all()                               # tail bytes stay in the row's place
    assert (rr * stride + (s & 15) + SEG - bb + READ_END[fmt] <= slot).all()  # decoder reads inside the slot
    per_tile = np.bincount(n // R, weights=(ce - al))
    assert per_tile.max() < 2**20                                 # one mbarrier transaction count per tile
    if fmt in ("Q4_K", "Q5_K", "W8A16_CHANNEL"):
        assert ((s & 15) == 0).all()


def check_plan(fmt, m, N, K, sms, occ):
    kc = qg.qgemv_chunk_k(fmt, m, K)
    assert kc > 0 and kc % (BLOCK[fmt][1]) == 0
    if kc < K:
        assert kc % 256 == 0
        first = qg.qgemv_plan_info(fmt, m, N, K, num_sms=sms, ctas_per_sm=occ)
        for c0 in range(0, K, kc):
            kw = min(kc, K - c0)
            p = qg.qgemv_plan_info_chunk(fmt, m, N, kw, num_sms=sms, ctas_per_sm=occ)
            if c0 == 0:
                assert {k: p[k] for k in first} == first   # the call's plan is its first chunk's
            check_chunked_plan(fmt, m, N, K, c0, kw, p)
        return
    p = qg.qgemv_plan_info(fmt, m, N, K, num_sms=sms, ctas_per_sm=occ)
    bb, be = BLOCK[fmt]
    nb = K // be
    RB = nb * bb
    total = N * RB
    assert p["row_bytes"] == RB
    R, S, slot, G = p["rows_per_tile"], p["stages"], p["stage_bytes"], p["team_warps"]
    assert 1 <= R <= N and 2 <= S <= 8
    assert slot % 128 == 0 and p["x_stage_bytes"] % 128 == 0 and p["red_bytes"] % 128 == 0
    assert BAR_BYTES + p["red_bytes"] + p["x_stage_bytes"] + S * slot == p["smem"] <= SMEM_CAP
    assert p["threads"] == 32 * (NC + 1)
    assert G in (1, 2, 4, 8) and NC % G == 0
    assert p["lanes"] == 32 * G if G > 1 else p["lanes"] in (4, 8, 16, 32)
    km = 16 if p["kernel_build"] == 10 else min(m, 8)  # rows the kernel build stages
    # 13: the 8-row build with row pairs (Q6_K only)
    assert p["kernel_build"] == 10 if km == 16 else p["kernel_build"] in (0, 1, 2, 3, 4, 5, 6, 7, 8, 13)
    if p["kernel_build"] == 13:
        assert fmt == "Q6_K" and m == 8 and G == 1
    if G > 1:  # reduction area: a counter and G*km partials per (slot, row)
        assert p["red_bytes"] >= 8 * R * 4 + 8 * R * G * km * 4
    assert p["num_tiles"] == -(-N // R)
    assert 1 <= p["grid"] <= p["num_tiles"]
    tiles = np.arange(p["num_tiles"], dtype=np.int64)
    r0 = tiles * R
    s = r0 * RB
    e = np.minimum(r0 + R, N) * RB
    rows = np.minimum(r0 + R, N) - r0
    al = s & ~15
    ce = np.minimum((e + 15) & ~15, total & ~15)
    assert (al >= 0).all() and (ce >= al).all() and (ce <= total).all()
    assert ((ce - al) % 16 == 0).all()
    assert (e - al <= slot).all()                  # tail bytes land inside the slot
    furthest = (s & 15) + (rows - 1) * RB + (RB - bb) + READ_END[fmt]
    assert (furthest <= slot).all()                # decoder reads stay inside the slot
    if fmt in ("Q4_K", "Q5_K", "W8A16_CHANNEL"):
        assert ((s & 15) == 0).all()               # 16-byte loads need aligned blocks


@pytest.mark.parametrize("fmt,N,K", _shapes())
def test_plans_keep_every_access_in_bounds(fmt, N, K):
    for m in (1, 3, 8, 9, 16):
        maxk = (qg.qgemv_max_k_w8a16(m) if fmt == "W8A16" else
                qg.qgemv_max_k_w8a16_channel(m) if fmt == "W8A16_CHANNEL" else qg.qgemv_max_k(fmt, m))
        if K > maxk:
            continue
        for sms, occ in ((152, 1), (152, 2), (152, 4), (10, 1)):
            check_plan(fmt, m, N, K, sms, occ)


def test_tuning_override_is_applied_and_cleared():
    try:
        qg.qgemv_tune_override(0, 3, 40, 2)
        p = qg.qgemv_plan_info("Q4_K", 1, 1000, 2560)
        assert (p["lanes"], p["rows_per_tile"], p["stages"]) == (8, 40, 2)
        check_plan("Q4_K", 1, 1000, 2560, 152, 1)
    finally:
        qg.qgemv_tune_override()
    p = qg.qgemv_plan_info("Q4_K", 1, 1000, 2560)
    assert p["rows_per_tile"] != 40 or p["stages"] != 2


def test_quantizer_grid_covers_blocks_exactly():
    # launch_quantize: 8 threads per 32-value block, 256-thread CTAs; threads past the last block
    # neither load nor store.
    for m in range(1, 17):
        for K in (32, 1024, 2560, 9728, 16384):
            nblocks = m * K // 32
            grid = -(-nblocks * 8 // 256)
            assert grid * 256 >= nblocks * 8 > (grid - 1) * 256


def test_single_row_build_choice():
    # single-row launches streaming >= 4 MB of weights use the streaming build (kind 0), others the
    # m-row kernel; m > 1 never uses the streaming build; the override forces either build
    small = qg.qgemv_plan_info("Q4_K", 1, 4096, 1024)
    big = qg.qgemv_plan_info("Q4_K", 1, 19456, 2560)
    multi = qg.qgemv_plan_info("Q4_K", 4, 19456, 2560)
    assert (small["kernel_build"], big["kernel_build"], multi["kernel_build"]) == (1, 0, 4)
    try:
        qg.qgemv_tune_override(kernel_build=2)
        assert qg.qgemv_plan_info("Q4_K", 1, 4096, 1024)["kernel_build"] == 0
        assert qg.qgemv_plan_info("Q4_K", 2, 4096, 1024)["kernel_build"] == 2
        qg.qgemv_tune_override(kernel_build=1)
        assert qg.qgemv_plan_info("Q4_K", 1, 19456, 2560)["kernel_build"] == 1
    finally:
        qg.qgemv_tune_override()


def test_medium_m_build_choice():
    # m = 9..16: the 16-row build where its activation staging fits, else the plan of the first of two
    # launches (8 rows, then m - 8)
    for m in (9, 12, 16):
        assert qg.qgemv_plan_info("Q4_K", m, 4096, 1024)["kernel_build"] == 10
        assert qg.qgemv_plan_info("Q8_0", m, 151936, 1024)["kernel_build"] == 10
    assert qg.qgemv_plan_info("Q6_K", 16, 2560, 9728)["kernel_build"] == 8
    assert qg.qgemv_plan_info("W8A16", 16, 7168, 8192)["kernel_build"] == 8


def test_row_pair_plans():
    # Q4_K at m = 4..8 with lane-row teams: tiles of two rows per team when that still gives most teams a
    # pair; the tuning hook forces pairs off (one row per team) or on
    def plan(m, N, K):
        return qg.qgemv_plan_info("Q4_K", m, N, K, num_sms=152, ctas_per_sm=1)
    try:
        for m in (4, 8):
            auto = plan(m, 19456, 2560)
            qg.qgemv_tune_pairs(2)
            off = plan(m, 19456, 2560)
            qg.qgemv_tune_pairs(0)
            assert auto["lanes"] == off["lanes"] == 8          # the row team shape never changes
            assert auto["rows_per_tile"] == 2 * off["rows_per_tile"] == 64
            check_plan("Q4_K", m, 19456, 2560, 152, 1)
        # not for m = 2 or 16, nor for the other formats
        for m in (2, 16):
            qg.qgemv_tune_pairs(1)
            forced = plan(m, 19456, 2560)
            qg.qgemv_tune_pairs(2)
            assert plan(m, 19456, 2560)["rows_per_tile"] == forced["rows_per_tile"]
            qg.qgemv_tune_pairs(0)
        qg.qgemv_tune_pairs(1)
        a = qg.qgemv_plan_info("Q6_K", 8, 2560, 9728, num_sms=152, ctas_per_sm=1)
        qg.qgemv_tune_pairs(2)
        b = qg.qgemv_plan_info("Q6_K", 8, 2560, 9728, num_sms=152, ctas_per_sm=1)
        assert a["rows_per_tile"] == b["rows_per_tile"]
    finally:
        qg.qgemv_tune_pairs(0)


def test_long_q6k_rows_take_half_team_tiles():
    # single-row Q6_K launches of multi-warp rows: tiles of half the teams and two ring slots (more CTAs per
    # SM, a more even spread of tiles); m > 1 and the other formats keep one row per team
    p = qg.qgemv_plan_info("Q6_K", 1, 2560, 9728, num_sms=152, ctas_per_sm=4)
    assert (p["team_warps"], p["rows_per_tile"], p["stages"]) == (2, 2, 2)
    assert p["smem"] * 4 <= SMEM_CAP
    check_plan("Q6_K", 1, 2560, 9728, 152, 4)
    assert qg.qgemv_plan_info("Q6_K", 2, 2560, 9728)["rows_per_tile"] == 4
    assert qg.qgemv_plan_info("W8A16", 1, 16384, 7168)["rows_per_tile"] == 4
    assert qg.qgemv_plan_info("Q6_K", 1, 151936, 2560)["rows_per_tile"] == 16


def test_q6k_row_pairs_take_their_own_build_at_m8_only():
    # the 8-row Q6_K launches of single-warp teams pair rows in a build of their own (kind 13); the
    # multi-warp rows (K = 9728) and the other row counts keep the plain m-row build
    lm = qg.qgemv_plan_info("Q6_K", 8, 151936, 2560)
    assert (lm["kernel_build"], lm["team_warps"]) == (13, 1)
    assert lm["rows_per_tile"] == 2 * 16  # two rows for each of the 16 lane teams of 16 lanes
    check_plan("Q6_K", 8, 151936, 2560, 152, 1)
    assert qg.qgemv_plan_info("Q6_K", 8, 2560, 9728)["kernel_build"] == 8
    for m in (1, 2, 4, 7):
        assert qg.qgemv_plan_info("Q6_K", m, 151936, 2560)["kernel_build"] in (0, m)
    assert qg.qgemv_plan_info("Q4_K", 8, 19456, 2560)["kernel_build"] == 8  # Q4_K pairs inside the 8-row build
