"""Compile the CPU oracle (plain C, gcc) into oracle/_build/liboracle.so.

The oracle is test infrastructure: this script builds the checker, it does not
put it on any product path.  Host-portable flags only (the same command builds
on x86_64 and aarch64).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "swiglu_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Build the shared library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -ffp-contract=off: no fused multiply-add, so every product is rounded to
    # fp64 before it is added (exact anyway for bf16/f32 operands).
    cmd = ["gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-fPIC", "-shared",
           "-ffp-contract=off", "-fno-fast-math", "-pthread",
           SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
