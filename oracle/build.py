"""Builds the CPU oracle (test infrastructure) into oracle/liboracle.so.

The flags keep binary32 arithmetic IEEE-exact: no fast-math and no
contraction of a*b+c into a fused multiply-add, on x86-64 and AArch64 alike.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-std=c99", "-O2", "-fno-fast-math", "-ffp-contract=off",
          "-fno-strict-aliasing", "-fPIC", "-shared", "-fvisibility=hidden"]


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
