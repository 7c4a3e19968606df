"""Compile the C oracle into ``oracle/liboracle.so`` (test infrastructure only).

Plain gcc, ``-O2`` without fast-math so that every double operation is IEEE and
in source order; OpenMP when the compiler has it (the loops over (sequence,
head) are independent, so threading does not change any result).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def compile_library(src: str, out: str, verbose: bool = False) -> str:
    """Compile one C source into a shared library at ``out``."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", src, "-o", out + ".tmp", "-lm"]
    r = None
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(out + ".tmp", out)
            if verbose:
                print(" ".join(cmd))
            return out
    raise RuntimeError("oracle build failed:\n" + r.stderr)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_library(SRC, LIB, verbose)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
