"""Compile the fp64 CPU oracle (plain C, OpenMP) into oracle/liboracle.so.

Test infrastructure only: the product library never links or loads it.
Flags keep IEEE semantics on every host (no fast-math, no FMA contraction),
so the oracle gives the same numbers on x86-64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ["layout.c", "attention.c", "accept.c"]
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    srcs = [os.path.join(HERE, s) for s in SOURCES]
    deps = srcs + [os.path.join(HERE, "simsd_oracle.h")]
    if not force and os.path.exists(LIB):
        lib_time = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= lib_time for d in deps):
            return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           "-o", tmp] + srcs + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
