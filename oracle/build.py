"""Compile the CPU oracle (plain C) into ``oracle/liboracle.so``.

Test infrastructure: the oracle is the independent checker of the CUDA path.
Flags: no FMA contraction and no fast-math, so every fl32 step in the C source
is one IEEE single-precision operation rounded to nearest even.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8q_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
          "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra"]


def build(src=SRC, out=LIB, extra=(), force=False, quiet=True):
    """Compile ``src`` into shared library ``out`` unless it is up to date."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src) and not extra):
        return out
    cmd = ["gcc", *CFLAGS, *extra, src, "-o", out, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + " ".join(cmd) + "\n" + res.stderr)
    if not quiet and res.stderr:
        sys.stderr.write(res.stderr)
    return out


if __name__ == "__main__":
    print(build(force=True, quiet=False))
