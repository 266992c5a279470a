"""Build the fp64 CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, -O2, no fast-math: the oracle keeps IEEE fp64 semantics and the
evaluation order written in oracle.c.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def compile_library(src: str, lib: str) -> str:
    """gcc one oracle source into a shared library, with the oracle's flags."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-Wextra", "-o", lib, src, "-lm"]
    subprocess.run(cmd, check=True)
    return lib


def build(force: bool = False) -> str:
    """The oracle library; ORACLE_LIB names another build of it instead (the
    test that plants mistakes in copies of the source uses this)."""
    other = os.environ.get("ORACLE_LIB")
    if other:
        return other
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_library(SRC, LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
