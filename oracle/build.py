"""Build the CPU oracle shared library (oracle/liboracle.so) with gcc.

Test infrastructure only: the product library never links or loads it.
Flags: -O2, no fast-math, floating-point contraction off (so a*b+c is two
rounded operations, as the activation-quantization reading requires), OpenMP
when the compiler supports it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bl_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter"]
    tmp = LIB + ".tmp.%d" % os.getpid()
    for extra in (["-fopenmp"], []):
        cmd = base + extra + [SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            if verbose:
                print(" ".join(cmd))
            return LIB
        if verbose:
            print(r.stderr, file=sys.stderr)
    raise RuntimeError("oracle build failed:\n" + r.stderr)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
