"""Build step for the CPU oracle (test infrastructure only).

Compiles ``fg_oracle.c`` with the host C compiler into ``_build/liboracle.so``
beside this file.  Plain C11 + POSIX threads, no architecture-specific flags,
so the same source builds on x86-64 and on Arm hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fg_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [cc, "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-D_POSIX_C_SOURCE=200809L", SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
