"""Compile the FP64 oracle (``oracle_fp64.c``) into ``oracle/_build/liboracle_fp64.so``.

Test infrastructure only: the product library never links or loads this.
OpenMP is used when the compiler accepts ``-fopenmp``; otherwise the oracle is
built single-threaded.  ``-ffp-contract=off`` keeps x86 and Arm results
identical (no fused multiply-adds chosen by the compiler).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle_fp64.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle_fp64.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]
    tmp = LIB + ".tmp%d" % os.getpid()
    for extra in (["-fopenmp"], []):
        cmd = base + extra + [SRC, "-o", tmp, "-lm"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode == 0:
            os.replace(tmp, LIB)
            if verbose:
                print(" ".join(cmd))
            return LIB
        if verbose:
            print(res.stderr, file=sys.stderr)
    raise RuntimeError("could not compile the oracle: " + res.stderr)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
