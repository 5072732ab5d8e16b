"""Compile the fp64 CPU oracles (attn_oracle.c, linear_attn_oracle.c) into
oracle/liboracle.so.

TEST INFRASTRUCTURE ONLY: the oracle is the parity checker for the CUDA path
and is never linked into, imported by or called from the product library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
SRC_LINEAR = os.path.join(HERE, "linear_attn_oracle.c")
SRCS = [SRC, SRC_LINEAR]
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Build liboracle.so if missing or older than its source; return its path."""
    if (not force and os.path.exists(LIB)
            and all(os.path.getmtime(LIB) >= os.path.getmtime(s) for s in SRCS)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    # No -ffast-math: the oracle must keep IEEE double semantics.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           *SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
