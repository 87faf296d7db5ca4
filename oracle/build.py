"""Build the CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, C11, -O2 with floating-point contraction disabled so that every
multiply and add rounds on its own, as the oracle's arithmetic is written.
OpenMP is used when the compiler supports it (rows of a decode step run in
parallel; results do not depend on the thread count).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fathom_oracle.c")
OUT = os.path.join(HERE, "liboracle.so")

FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= os.path.getmtime(SRC):
        return OUT
    tmp = OUT + ".tmp%d" % os.getpid()
    cmd = ["gcc", *FLAGS, "-fopenmp", SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP runtime: build single-threaded
        cmd = ["gcc", *FLAGS, SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
