"""Compile the C oracle into ``oracle/liboracle_fp8fg.so`` with gcc.

Test infrastructure only: the oracle is the CPU restatement that the tests,
the smoke check and the benchmark's CPU-baseline leg compare against.  IEEE
single-precision division and multiplication must be kept exactly, so the
build uses no fast-math flags and forbids FMA contraction.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8fg_oracle.c")
LIB = os.path.join(HERE, "liboracle_fp8fg.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fexcess-precision=standard", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
