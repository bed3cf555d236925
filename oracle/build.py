"""Compile the C oracle into ``oracle/libkvoracle.so`` (test infrastructure).

Plain gcc, fp64 loops, floating-point contraction off so that the oracle
rounds the same way on x86-64 and on aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvoracle.c")
LIB = os.path.join(HERE, "libkvoracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-Wno-maybe-uninitialized"]


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile ``src`` into the shared library ``out`` and return its path."""
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def needs_build(src: str = SRC, out: str = LIB) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)


if __name__ == "__main__":
    print(build(*sys.argv[1:2]))
