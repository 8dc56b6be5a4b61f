"""Compile the CPU oracle (test infrastructure) into oracle/libozk_oracle.so.

Plain gcc, no CUDA.  -ffp-contract=off keeps every product and sum separately
rounded, which the compensated reference relies on.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ozk_oracle.c")
LIB = os.path.join(HERE, "libozk_oracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(
        os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "ozk_oracle.h"))
    ):
        return LIB
    cmd = [
        os.environ.get("CC", "gcc"), "-O2", "-std=gnu11", "-fopenmp", "-ffp-contract=off",
        "-fno-fast-math", "-fPIC", "-shared", "-Wall", "-Wextra", "-o", LIB, SRC, "-lm",
    ]
    subprocess.run(cmd, check=True)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
