"""Build the CPU oracle library (test infrastructure only).

Compiles ``qlin_oracle.c`` with gcc into ``liborc.so`` beside this file.  The
flags keep every binary32 operation a single IEEE-754 operation: no
fast-math, no FMA contraction.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qlin_oracle.c")
LIB = os.path.join(HERE, "liborc.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
          "-fno-fast-math", "-ffp-contract=off", "-fno-builtin-nearbyintf",
          "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    """Compile the oracle if the source is newer than the library; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
