"""Compile the C oracle into ``oracle/_build/libmx_oracle.so`` with gcc.

Test infrastructure: the oracle is built so that tests, the smoke check and the
benchmark's CPU-baseline leg can call it.  Building it does not make the CUDA
library depend on it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mx_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmx_oracle.so")


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -O2 without -ffast-math: the oracle relies on IEEE double semantics and
    # on nearbyint() rounding ties to even.  OpenMP only spreads independent
    # rows / columns over host threads (oracle_set_threads); where the
    # compiler has no OpenMP runtime the oracle is built sequential.
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    if subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True).returncode != 0:
        subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
