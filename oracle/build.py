"""Compile the CPU oracle (moe_oracle.c) into liboracle.so beside this file.

Test infrastructure: the oracle is built here so the tests, the smoke check and the
benchmark's CPU-baseline leg can load it; the product path never does.

Plain ``gcc -O2 -fopenmp``: no fast-math, no host-specific tuning, so it builds and gives
the same results on x86_64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def compile_oracle(src=SRC, out=LIB, extra=()):
    """Build ``src`` into the shared library ``out``; return ``out``."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           "-Werror", *extra, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def up_to_date(src=SRC, out=LIB):
    return os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src)


if __name__ == "__main__":
    print(compile_oracle(*sys.argv[1:2]))
