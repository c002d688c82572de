"""Mutation test of the oracle's pins: plausible mistakes planted in copies of oracle.c must each make
at least one pin fail, and the unmodified copy must pass.  CPU only (gcc); the mutants live in a
temporary directory and are loaded through ORACLE_LIB_OVERRIDE by a child pytest run.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text in oracle.c, planted replacement)
MUTANTS = [
    ("k-quant nibbles swapped", "(qs[32 * g + r] & 0x0F) : (qs[32 * g + r - 32] >> 4)",
     "(qs[32 * g + r] >> 4) : (qs[32 * g + r - 32] & 0x0F)"),
    ("k-quant min term sign", "- dmin * (double)field[8 + j]", "+ dmin * (double)field[8 + j]"),
    ("k-quant min read from the scale field", "- dmin * (double)field[8 + j]", "- dmin * (double)field[j]"),
    ("k-quant sub-block index", "int j = e / 32;", "int j = e / 64;"),
    ("k-quant scale field width", "for (int k = 0; k < 6; ++k) v |= bit_at(b + 4, 6 * f + k) << k;",
     "for (int k = 0; k < 5; ++k) v |= bit_at(b + 4, 6 * f + k) << k;"),
    ("q4k qs offset", "low_nibble_code(b + 16, e)", "low_nibble_code(b + 12, e)"),
    ("q6k bias", "(double)(q - 32)", "(double)(q - 31)"),
    ("q6k sub-scale index", "sc[e / 16]", "sc[e / 32]"),
    ("q6k high-bit shift", "(qh[32 * h + t] >> (2 * k)) & 3", "(qh[32 * h + t] >> k) & 3"),
    ("q6k low nibbles swapped", "(ql[64 * h + r] & 0x0F) : (ql[64 * h + r - 64] >> 4)",
     "(ql[64 * h + r] >> 4) : (ql[64 * h + r - 64] & 0x0F)"),
    ("q80 code offset", "(int8_t)b[2 + j]", "(int8_t)b[1 + j]"),
    ("quantizer ties to even", "roundf(xb[j] / d32)", "rintf(xb[j] / d32)"),
    ("quantizer clamp -128", "if (r < -127.0f) r = -127.0f;", "if (r < -128.0f) r = -128.0f;"),
    ("quantizer scale 1/128", "float d32 = amax / 127.0f;", "float d32 = amax / 128.0f;"),
    ("s without the scale", "float sp = dfl * (float)sum;", "float sp = (float)sum;"),
    ("fp16 ties away from zero", "(rem == 0x1000u && (h & 1u))", "(rem == 0x1000u)"),
    ("activation row ignored", "const double* xi = xhat + (size_t)i * K;", "const double* xi = xhat;"),
    ("q8_1 code offset", "(double)(int8_t)blk[4 + j]", "(double)(int8_t)blk[3 + j]"),
    ("q5k high-bit index", "int hi = (qh[e % 32] >> (e / 32)) & 1;", "int hi = (qh[e % 32] >> (e / 64)) & 1;"),
    ("q5k high-bit weight", "int q = low_nibble_code(qs, e) + 16 * hi;", "int q = low_nibble_code(qs, e) + 8 * hi;"),
    ("q5k qs offset", "const uint8_t* qs = b + 48;", "const uint8_t* qs = b + 16;"),
]


def _build(src_text, path):
    c = path + ".c"
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                    "-fexcess-precision=standard", c, "-o", path, "-lm"], check=True)
    return path


def _pins_pass(lib_path):
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=lib_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode == 0, r.stdout[-400:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    text = open(SRC).read()
    for name, old, new in MUTANTS:
        assert text.count(old) == 1, f"mutation site not unique or missing: {name}"
    control = _build(text, str(tmp_path / "control.so"))
    libs = [_build(text.replace(old, new), str(tmp_path / f"m{i}.so")) for i, (_, old, new) in enumerate(MUTANTS)]
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(_pins_pass, [control] + libs))
    ok, out = results[0]
    assert ok, f"unmodified oracle copy fails its pins:\n{out}"
    survivors = [MUTANTS[i][0] for i, (passed, _) in enumerate(results[1:]) if passed]
    assert not survivors, f"planted mistakes no pin catches: {survivors}"
