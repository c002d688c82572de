"""Independent block decoder and packer used to pin the oracle (test helper, numpy only).

Written from the block definitions in the opposite direction to the oracle: the oracle maps each element
to its byte/nibble, this module walks each BYTE (and each bit of the scale bit string) and says which
element(s) it feeds.  fp16 fields are decoded with numpy's own binary16 type, not the oracle's decoder.
A mistake in either side's index arithmetic (swapped nibbles, wrong group stride, wrong field offset)
makes the two disagree.
"""
import numpy as np

BLOCK = {"Q4_K": (144, 256), "Q5_K": (176, 256), "Q6_K": (210, 256), "Q8_0": (34, 32)}


def _f16(b: np.ndarray, off: int) -> float:
    return float(np.frombuffer(bytes(b[off:off + 2]), dtype="<f2")[0])


def q4k_fields(blk: np.ndarray):
    """(d, dmin, sc[8], mn[8], q[256]) decoded byte-wise."""
    d, dmin = _f16(blk, 0), _f16(blk, 2)
    bits = np.unpackbits(blk[4:16], bitorder="little").astype(np.int64)  # bit t of the 96-bit string
    fields = [int(sum(int(bits[6 * f + k]) << k for k in range(6))) for f in range(16)]
    q = np.full(256, -1, dtype=np.int64)
    for p in range(128):  # qs byte p
        g, t = divmod(p, 32)
        byte = int(blk[16 + p])
        q[64 * g + t] = byte & 0xF
        q[64 * g + 32 + t] = byte >> 4
    assert (q >= 0).all()
    return d, dmin, fields[:8], fields[8:], q


def q5k_fields(blk: np.ndarray):
    """(d, dmin, sc[8], mn[8], q[256]) decoded byte-wise: the Q4_K header and nibbles (qs at byte 48)
    plus one high bit per element from the 32 qh bytes at byte 16."""
    d, dmin = _f16(blk, 0), _f16(blk, 2)
    bits = np.unpackbits(blk[4:16], bitorder="little").astype(np.int64)
    fields = [int(sum(int(bits[6 * f + k]) << k for k in range(6))) for f in range(16)]
    q = np.full(256, -1, dtype=np.int64)
    for p in range(128):  # qs byte p
        g, t = divmod(p, 32)
        byte = int(blk[48 + p])
        q[64 * g + t] = byte & 0xF
        q[64 * g + 32 + t] = byte >> 4
    for t in range(32):  # qh byte t: bit j belongs to element 32j + t
        byte = int(blk[16 + t])
        for j in range(8):
            q[32 * j + t] += 16 * ((byte >> j) & 1)
    assert (q >= 0).all()
    return d, dmin, fields[:8], fields[8:], q


def q6k_fields(blk: np.ndarray):
    """(d, sc[16], q[256]) decoded byte-wise."""
    low = np.full(256, -1, dtype=np.int64)
    high = np.full(256, -1, dtype=np.int64)
    for p in range(128):  # ql byte p
        h, t = divmod(p, 64)
        byte = int(blk[p])
        low[128 * h + t] = byte & 0xF
        low[128 * h + 64 + t] = byte >> 4
    for p in range(64):  # qh byte p
        h, t = divmod(p, 32)
        byte = int(blk[128 + p])
        for k in range(4):
            high[128 * h + 32 * k + t] = (byte >> (2 * k)) & 3
    assert (low >= 0).all() and (high >= 0).all()
    sc = blk[192:208].view(np.int8).astype(np.int64)
    return _f16(blk, 208), sc, low + 16 * high


def dense_rows(fmt: str, W: np.ndarray, N: int, K: int) -> np.ndarray:
    bb, be = BLOCK[fmt]
    nb = K // be
    W = W.reshape(N, nb, bb)
    out = np.empty((N, K), dtype=np.float64)
    for n in range(N):
        for b in range(nb):
            blk = W[n, b]
            seg = out[n, b * be:(b + 1) * be]
            if fmt in ("Q4_K", "Q5_K"):
                d, dmin, sc, mn, q = q4k_fields(blk) if fmt == "Q4_K" else q5k_fields(blk)
                for e in range(256):
                    seg[e] = d * sc[e // 32] * q[e] - dmin * mn[e // 32]
            elif fmt == "Q6_K":
                d, sc, q = q6k_fields(blk)
                for e in range(256):
                    seg[e] = d * sc[e // 16] * (q[e] - 32)
            else:
                d = _f16(blk, 0)
                seg[:] = d * blk[2:34].view(np.int8).astype(np.float64)
    return out


def dense_act(xq: np.ndarray, m: int, K: int) -> np.ndarray:
    nb = K // 32
    xq = xq.reshape(m, nb, 36)
    out = np.empty((m, K), dtype=np.float64)
    for i in range(m):
        for b in range(nb):
            out[i, 32 * b:32 * b + 32] = _f16(xq[i, b], 0) * xq[i, b, 4:36].view(np.int8)
    return out


# ------------------------------------------------------------------------------------------------------
# Packers (element values -> bytes), for constructing special blocks in tests.

def f16_bytes(v: float) -> bytes:
    return np.array([v], dtype="<f2").tobytes()


def pack_q4k(d: float, dmin: float, sc, mn, q) -> np.ndarray:
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.frombuffer(f16_bytes(d), np.uint8)
    blk[2:4] = np.frombuffer(f16_bytes(dmin), np.uint8)
    bits = np.zeros(96, dtype=np.uint8)
    for f, v in enumerate(list(sc) + list(mn)):
        assert 0 <= v < 64
        for k in range(6):
            bits[6 * f + k] = (v >> k) & 1
    blk[4:16] = np.packbits(bits, bitorder="little")
    for p in range(128):
        g, t = divmod(p, 32)
        lo, hi = int(q[64 * g + t]), int(q[64 * g + 32 + t])
        assert 0 <= lo < 16 and 0 <= hi < 16
        blk[16 + p] = lo | (hi << 4)
    return blk


def pack_q5k(d: float, dmin: float, sc, mn, q) -> np.ndarray:
    blk = np.zeros(176, dtype=np.uint8)
    blk[0:2] = np.frombuffer(f16_bytes(d), np.uint8)
    blk[2:4] = np.frombuffer(f16_bytes(dmin), np.uint8)
    bits = np.zeros(96, dtype=np.uint8)
    for f, v in enumerate(list(sc) + list(mn)):
        assert 0 <= v < 64
        for k in range(6):
            bits[6 * f + k] = (v >> k) & 1
    blk[4:16] = np.packbits(bits, bitorder="little")
    q = [int(v) for v in q]
    assert all(0 <= v < 32 for v in q)
    for t in range(32):
        blk[16 + t] = sum(((q[32 * j + t] >> 4) & 1) << j for j in range(8))
    for p in range(128):
        g, t = divmod(p, 32)
        blk[48 + p] = (q[64 * g + t] & 0xF) | ((q[64 * g + 32 + t] & 0xF) << 4)
    return blk


def pack_q6k(d: float, sc, q) -> np.ndarray:
    blk = np.zeros(210, dtype=np.uint8)
    q = [int(v) for v in q]
    assert all(0 <= v < 64 for v in q)
    for p in range(128):
        h, t = divmod(p, 64)
        blk[p] = (q[128 * h + t] & 0xF) | ((q[128 * h + 64 + t] & 0xF) << 4)
    for p in range(64):
        h, t = divmod(p, 32)
        blk[128 + p] = sum(((q[128 * h + 32 * k + t] >> 4) & 3) << (2 * k) for k in range(4))
    blk[192:208] = np.array(sc, dtype=np.int8).view(np.uint8)
    blk[208:210] = np.frombuffer(f16_bytes(d), np.uint8)
    return blk


def pack_q80(d: float, q) -> np.ndarray:
    blk = np.zeros(34, dtype=np.uint8)
    blk[0:2] = np.frombuffer(f16_bytes(d), np.uint8)
    blk[2:34] = np.array(q, dtype=np.int8).view(np.uint8)
    return blk


def pack_q8_1(d: float, s: float, q) -> np.ndarray:
    blk = np.zeros(36, dtype=np.uint8)
    blk[0:2] = np.frombuffer(f16_bytes(d), np.uint8)
    blk[2:4] = np.frombuffer(f16_bytes(s), np.uint8)
    blk[4:36] = np.array(q, dtype=np.int8).view(np.uint8)
    return blk
