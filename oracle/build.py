"""Build the C part of the CPU oracle (test infrastructure, never the product path).

Compiles ``mx_oracle.c`` into ``oracle/_build/libmx_oracle.so`` with plain gcc.
``-ffp-contract=off`` keeps the fp32 Hadamard sequence unfused on every host
(gcc contracts a*b+c by default on aarch64).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mx_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmx_oracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    base = ["gcc", "-std=gnu11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", SRC, "-o", tmp, "-lm"]
    # OpenMP only splits independent rows across threads; without it the
    # oracle computes the same bytes serially.
    if subprocess.run(base + ["-fopenmp"], capture_output=True).returncode != 0:
        subprocess.run(base, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
