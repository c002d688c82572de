"""Synthetic decode-sweep workloads: shapes, formats and seeds (no arithmetic of the method).

A workload is an ordered list of operations, the way one decode token walks the layer stack:
``QuantOp`` quantizes one activation input once, every ``GemvOp`` that reads that input follows it.
Each weight matrix and each activation row has its own seeded stream.

Shapes (N = output rows, K = input length), one decode token (m = 1 unless stated):
  dense-q4k-256x1024 : one Q4_K GEMV, N=256, K=1024.
  dense-0.6b-class   : 28 layers x {q 2048x1024, k 1024x1024, v 1024x1024, o 1024x2048, gate 3072x1024,
                       up 3072x1024 (Q4_K), down 1024x3072 (Q6_K)} + lm_head 151936x1024 (Q8_0).
  dense-4b-class     : 36 layers x {qkv 6144x2560, o 2560x4096, gate 9728x2560, up 9728x2560 (Q4_K),
                       down 2560x9728 (Q6_K)} + lm_head 151936x2560 (Q6_K).
  dense-4b-class-mM  : the same with m in {2, 4, 8, 16} activation rows per call.
  w8a16-large        : 20 layers x {16384x7168, 7168x16384} Q8_0 weights against bf16 activations.
"""
from dataclasses import dataclass, field
from typing import List, Tuple

# format name -> (bytes per block, elements per block)
FORMATS = {"Q4_K": (144, 256), "Q5_K": (176, 256), "Q6_K": (210, 256), "Q8_0": (34, 32)}
FMT_CODE = {"Q4_K": 1, "Q6_K": 2, "Q8_0": 3, "Q5_K": 5}

BASE_SEED = 0x5EED_0F_DEC0DE


@dataclass
class QuantOp:
    input: str  # activation input name
    K: int


@dataclass
class GemvOp:
    name: str
    fmt: str  # "Q4_K" | "Q6_K" | "Q8_0"
    N: int
    K: int
    input: str
    w8a16: bool = False

    @property
    def weight_bytes(self) -> int:
        bb, be = FORMATS[self.fmt]
        return self.N * (self.K // be) * bb


@dataclass
class Workload:
    name: str
    m: int
    ops: List[object] = field(default_factory=list)
    seed: int = BASE_SEED

    @property
    def gemvs(self) -> List[GemvOp]:
        return [o for o in self.ops if isinstance(o, GemvOp)]

    @property
    def quants(self) -> List[QuantOp]:
        return [o for o in self.ops if isinstance(o, QuantOp)]

    @property
    def weight_bytes(self) -> int:
        return sum(g.weight_bytes for g in self.gemvs)

    def inputs(self) -> List[Tuple[str, int]]:
        """Distinct activation inputs (name, K) in first-use order."""
        seen, out = set(), []
        for o in self.ops:
            if isinstance(o, GemvOp) and o.input not in seen:
                seen.add(o.input)
                out.append((o.input, o.K))
        return out


def _tag(s: str) -> int:
    """Stable 64-bit tag of a tensor name (FNV-1a)."""
    h = 0xCBF29CE484222325
    for ch in s.encode():
        h = ((h ^ ch) * 0x100000001B3) & (2**64 - 1)
    return h


def weight_seed(wl: Workload, op: GemvOp) -> int:
    from . import derive
    return derive(wl.seed, _tag(wl.name.split("-m")[0]), _tag("W:" + op.name))


def input_seed(wl: Workload, input_name: str, row: int) -> int:
    from . import derive
    return derive(wl.seed, _tag(wl.name.split("-m")[0]), _tag("x:" + input_name), row)


def _single() -> Workload:
    wl = Workload("dense-q4k-256x1024", 1)
    wl.ops = [QuantOp("x", 1024), GemvOp("w", "Q4_K", 256, 1024, "x")]
    return wl


def _dense_06b() -> Workload:
    wl = Workload("dense-0.6b-class", 1)
    H, I = 1024, 3072
    for L in range(28):
        a, o, f, d = f"l{L}.attn_in", f"l{L}.o_in", f"l{L}.mlp_in", f"l{L}.down_in"
        wl.ops += [QuantOp(a, H),
                   GemvOp(f"l{L}.q", "Q4_K", 2048, H, a),
                   GemvOp(f"l{L}.k", "Q4_K", 1024, H, a),
                   GemvOp(f"l{L}.v", "Q4_K", 1024, H, a),
                   QuantOp(o, 2048),
                   GemvOp(f"l{L}.o", "Q4_K", H, 2048, o),
                   QuantOp(f, H),
                   GemvOp(f"l{L}.gate", "Q4_K", I, H, f),
                   GemvOp(f"l{L}.up", "Q4_K", I, H, f),
                   QuantOp(d, I),
                   GemvOp(f"l{L}.down", "Q6_K", H, I, d)]
    wl.ops += [QuantOp("lm_head_in", H), GemvOp("lm_head", "Q8_0", 151936, H, "lm_head_in")]
    return wl


def _dense_4b(m: int = 1) -> Workload:
    wl = Workload("dense-4b-class" if m == 1 else f"dense-4b-class-m{m}", m)
    H, I = 2560, 9728
    for L in range(36):
        a, o, f, d = f"l{L}.attn_in", f"l{L}.o_in", f"l{L}.mlp_in", f"l{L}.down_in"
        wl.ops += [QuantOp(a, H),
                   GemvOp(f"l{L}.qkv", "Q4_K", 6144, H, a),
                   QuantOp(o, 4096),
                   GemvOp(f"l{L}.o", "Q4_K", H, 4096, o),
                   QuantOp(f, H),
                   GemvOp(f"l{L}.gate", "Q4_K", I, H, f),
                   GemvOp(f"l{L}.up", "Q4_K", I, H, f),
                   QuantOp(d, I),
                   GemvOp(f"l{L}.down", "Q6_K", H, I, d)]
    wl.ops += [QuantOp("lm_head_in", H), GemvOp("lm_head", "Q6_K", 151936, H, "lm_head_in")]
    return wl


def _w8a16() -> Workload:
    wl = Workload("w8a16-large", 1)
    for L in range(20):
        a, b = f"l{L}.up_in", f"l{L}.down_in"
        wl.ops += [GemvOp(f"l{L}.up", "Q8_0", 16384, 7168, a, w8a16=True),
                   GemvOp(f"l{L}.down", "Q8_0", 7168, 16384, b, w8a16=True)]
    return wl


WORKLOADS = {
    "dense-q4k-256x1024": _single,
    "dense-0.6b-class": _dense_06b,
    "dense-4b-class": lambda: _dense_4b(1),
    "dense-4b-class-m2": lambda: _dense_4b(2),
    "dense-4b-class-m4": lambda: _dense_4b(4),
    "dense-4b-class-m8": lambda: _dense_4b(8),
    "dense-4b-class-m16": lambda: _dense_4b(16),
    "w8a16-large": _w8a16,
}
