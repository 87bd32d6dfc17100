"""Build the CPU oracle (plain C, OpenMP) into oracle/_build/liboracle.so.

Test infrastructure: only tests/, __graft_entry__ and bench.py's CPU
baseline leg use the library this builds.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liboracle.so")
SOURCES = [os.path.join(HERE, "oracle.c")]
HEADERS = [os.path.join(HERE, "oracle.h")]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in SOURCES + HEADERS + [__file__])


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its sources."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB + ".tmp%d" % os.getpid()
    # -ffp-contract=off: no fused multiply-add, so x86 and Arm give the same bits.
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp] + SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
