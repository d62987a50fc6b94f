"""Builds the FP64 CPU oracle (test infrastructure) into oracle/liboracle_vcd.so.

Plain C99 compiled with gcc. ``-ffp-contract=off`` keeps every product and sum
rounded as written, so the oracle gives the same doubles on x86-64 and AArch64.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vcd_oracle.c")
LIB = os.path.join(HERE, "liboracle_vcd.so")

CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def compile_oracle(src=SRC, out=LIB, extra=(), werror=True):
    """Compile ``src`` into the shared library ``out``; returns ``out``."""
    cmd = ["gcc", *CFLAGS, *(["-Werror"] if werror else []), *extra, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force=False):
    """Build the oracle library if it is missing or older than its source."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        compile_oracle()
    return LIB


if __name__ == "__main__":
    print(build(force=True))
