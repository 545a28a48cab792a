"""Compile the float64 CPU oracle (hc_oracle.c) into oracle/libhc_oracle.so.

Test infrastructure only: the library path never loads what this builds.
Plain gcc, no architecture-specific flags, so the same source builds on x86-64
and on aarch64.  Floating-point contraction is off so that every double
operation in the oracle rounds exactly as written.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hc_oracle.c")
LIB = os.path.join(HERE, "libhc_oracle.so")


def build(force: bool = False, openmp: bool = True) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra"]
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = base + (["-fopenmp"] if openmp else []) + [SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and openmp:
        cmd = base + [SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
