"""Build the CPU oracle (plain C, binary64) into oracle/libdv_oracle.so.

Test infrastructure: compiled by ``__graft_entry__.build()`` so that the test
suite can load it; nothing on the product path links or loads it.
Floating-point contraction is off so x86-64 and aarch64 builds give the same
bits.
"""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dv_oracle.c")
LIB = os.path.join(HERE, "libdv_oracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
