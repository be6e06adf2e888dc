"""Compile the CPU oracle into ``oracle/_build/liboracle.so``.

Test infrastructure: the oracle is built next to the product so that tests,
the smoke check and the benchmark's CPU-baseline leg can load it.  Building
the checker is not using it; nothing on the product path loads the result.

Flags: ``-O2 -ffp-contract=off -fno-fast-math`` so that every FP32 step is
one IEEE-754 binary32 operation with no fused multiply-add, identically on
x86-64 and aarch64 (gcc contracts to FMA by default on aarch64).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4kv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", LIB + ".tmp", SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
