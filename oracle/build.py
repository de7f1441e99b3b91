"""Compile the C oracle into ``oracle/liboracle.so`` with gcc.

Test infrastructure: the oracle is the independent CPU definition the CUDA
library is checked against.  Flags keep every fp32 operation a single IEEE
rounding: no FMA contraction, no fast-math, no host-specific instruction set.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fno-strict-aliasing", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(
                os.path.join(HERE, "moe_oracle.h"))):
        return LIB
    tmp = LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
