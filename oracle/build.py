"""Builds the CPU oracle's shared library with gcc.

Test infrastructure: the oracle is compiled on every machine that runs the
tests (x86_64 here, aarch64 on the GPU host), with FMA contraction and fast
math switched off so that each float expression is one IEEE binary32
operation.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "kvq_oracle.c")
HEADER = os.path.join(HERE, "kvq_oracle.h")
LIBRARY = os.path.join(HERE, "_build", "libkvq_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-Wall", "-Wextra", "-Werror",
          "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compiles oracle/kvq_oracle.c into oracle/_build/libkvq_oracle.so."""
    os.makedirs(os.path.dirname(LIBRARY), exist_ok=True)
    newest = max(os.path.getmtime(SOURCE), os.path.getmtime(HEADER),
                 os.path.getmtime(__file__))
    if not force and os.path.exists(LIBRARY) and os.path.getmtime(LIBRARY) >= newest:
        return LIBRARY
    tmp = LIBRARY + ".tmp.%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, SOURCE, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True))
