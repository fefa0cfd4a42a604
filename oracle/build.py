"""Compile the CPU oracle (plain C) into oracle/libvc_oracle.so.

Test infrastructure: the product path never loads this library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vc_oracle.c")
LIB = os.path.join(HERE, "libvc_oracle.so")


def compile_c(src: str, out: str) -> str:
    """Compile one C source into a shared library with the oracle's flags."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", src, "-o", out, "-lm"]
    subprocess.check_call(cmd)
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".%d.tmp" % os.getpid()
    compile_c(SRC, tmp)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
