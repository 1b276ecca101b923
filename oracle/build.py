"""Build the oracle's C core into oracle/_moe4_oracle.so (test infrastructure only).

The flags matter: -ffp-contract=off keeps every multiply and add a separate binary32 operation,
and no -ffast-math keeps IEEE semantics (signed zeros, exact comparisons, no reassociation).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe4_oracle.c")
LIB = os.path.join(HERE, "_moe4_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
