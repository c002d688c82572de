"""Compile the oracle (plain C, fp64, host only) into a shared library next to its source.

Test infrastructure: built by the package build step so the checker exists on every machine, but only
the tests, the smoke check and the benchmark's CPU-baseline leg load it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-add contraction, so every fp32 step of the quantizer is one
    # IEEE operation on both x86-64 and aarch64.
    cmd = ["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-fexcess-precision=standard", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB
