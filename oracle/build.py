"""Compile the C oracle into ``oracle/liboracle_fp8.so`` (test infrastructure).

Plain gcc, no CUDA: the oracle is host code only.  ``-ffp-contract=off`` keeps
every multiply and add separately rounded on both x86-64 and AArch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "liboracle_fp8.so")
SRC = [os.path.join(HERE, "fp8_oracle.c")]


def command():
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-o", LIB] + SRC + ["-lm"]


def start():
    """Start the compile and return the Popen (lets callers overlap builds)."""
    return subprocess.Popen(command(), stdout=subprocess.PIPE, stderr=subprocess.STDOUT)


def build():
    p = start()
    out, _ = p.communicate()
    if p.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + out.decode(errors="replace"))
    return LIB


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in SRC + [os.path.join(HERE, "fp8_oracle.h")])


if __name__ == "__main__":
    print(build())
    sys.exit(0)
