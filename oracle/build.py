"""Compile the CPU oracle (plain C, OpenMP) into oracle/libnf4_oracle.so.

Test infrastructure only: the test suite, the smoke check and the benchmark's CPU
baseline load the result.  Run as ``python oracle/build.py``.
"""
import hashlib
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nf4_oracle.c")
LIB = os.path.join(HERE, "libnf4_oracle.so")

# -ffp-contract=off: every fp32 multiply/add is one IEEE operation (no fused contraction),
# which the oracle's fp32 steps (normalisation, double quantization, dequantization) rely on.
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


STAMP = LIB + ".stamp"


def _digest() -> str:
    with open(SRC, "rb") as f:
        return hashlib.sha256(" ".join(CFLAGS).encode() + f.read()).hexdigest()


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == _digest():
                return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_digest())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
