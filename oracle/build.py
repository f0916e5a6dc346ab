"""Compile the CPU oracle (plain C) into a shared library.

TEST INFRASTRUCTURE: the oracle is built so that the tests, the smoke check and
the benchmark's CPU baseline can run it; the GPU library never links or loads it.

The flags keep the C compiler from changing the arithmetic the pages describe:
no contraction of a multiply and an add into one rounding, no fast-math, and no
auto-vectorisation (which would reorder the double running sums).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vqx_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libvqx_oracle.so")

CFLAGS = [
    "-O2",
    "-std=c11",
    "-fPIC",
    "-shared",
    "-ffp-contract=off",
    "-fno-fast-math",
    "-fno-tree-vectorize",
    "-fexcess-precision=standard",
]


def build_oracle(src=SRC, out=LIB, force=False):
    """Compile ``src`` into ``out`` (skipped when ``out`` is newer than ``src``)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
