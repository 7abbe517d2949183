"""Build liboracle.so (the fp64 CPU oracle) with the host C compiler.

Test infrastructure: the oracle is what the CUDA library is checked against.
Plain C11, no SIMD intrinsics, no fast-math, no FMA contraction, so that the
same source gives the same results on x86_64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "liboracle.so")
SRC = [os.path.join(HERE, "oracle.c")]


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/liboracle.so; returns the library path."""
    newest_src = max(os.path.getmtime(p) for p in SRC + [os.path.join(HERE, "oracle.h")])
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest_src:
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-std=c11", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp] + SRC + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
