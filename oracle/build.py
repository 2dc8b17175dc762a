"""Builds the CPU oracle (test infrastructure) into oracle/libkvq_oracle.so.

Plain gcc, no CUDA. Flags keep binary32 semantics literal: no contraction of
a*b+c into a fused multiply-add (GCC contracts by default in GNU mode, and
always on AArch64), no fast-math, gradual underflow.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "kvq_oracle.c")
LIBRARY = os.path.join(HERE, "libkvq_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-Werror"]


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    stale = (not os.path.exists(LIBRARY)
             or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))
    if force or stale:
        tmp = LIBRARY + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, SOURCE, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True))
