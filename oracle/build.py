"""Build the CPU oracle library (test infrastructure) in-tree with gcc + OpenMP.

Floating-point contraction is off so that x86 and Arm hosts give the same bits.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(HERE, "libpporacle.so")
SRC = ["pp_oracle.c", "pp_oracle.h"]


def cmd():
    return ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-std=c11", os.path.join(HERE, "pp_oracle.c"), "-o", SO, "-lm"]


def stale():
    if not os.path.exists(SO):
        return True
    t = os.path.getmtime(SO)
    return any(os.path.getmtime(os.path.join(HERE, f)) > t for f in SRC)


def build(force=False):
    if force or stale():
        subprocess.check_call(cmd())
    return SO


if __name__ == "__main__":
    build(force=True)
