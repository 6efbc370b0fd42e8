"""Build the CPU oracle (plain C, binary64) into oracle/libdv_oracle.so.

Test infrastructure: compiled by ``__graft_entry__.build()`` so that the test
suite can load it; nothing on the product path links or loads it.
Floating-point contraction is off so x86-64 and aarch64 builds give the same
bits.

A second library, oracle/libdv_oracle_omp.so, is the same source built with
OpenMP: the loops over independent output elements run on every host core
(each element still one plain loop in the same order, so the results are the
same bits).  It exists to time the CPU baseline on all cores; if the compiler
has no OpenMP it is skipped and ``build_omp`` returns None.
"""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dv_oracle.c")
LIB = os.path.join(HERE, "libdv_oracle.so")
LIB_OMP = os.path.join(HERE, "libdv_oracle_omp.so")

_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall",
          "-Wextra"]


def _compile(out: str, extra) -> None:
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *_FLAGS, *extra, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    os.replace(tmp, out)


def _fresh(lib: str) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    if force or not _fresh(LIB):
        _compile(LIB, ["-Wno-unknown-pragmas"])
    build_omp(force)
    return LIB


def build_omp(force: bool = False):
    """Path of the OpenMP build, or None when the compiler cannot make it."""
    if not force and _fresh(LIB_OMP):
        return LIB_OMP
    try:
        _compile(LIB_OMP, ["-fopenmp"])
    except (subprocess.CalledProcessError, OSError):
        return None
    return LIB_OMP


if __name__ == "__main__":
    print(build(force="--force" in sys.argv), build_omp())
