"""Compile the CPU oracle (test infrastructure) into oracle/_build/libkvq_oracle.so.

Plain gcc, -O2, no fast-math and no FMA contraction, so that every fp32
division and fp64 operation is the IEEE one the oracle's source states.
OpenMP is used when the compiler supports it (only to run independent rows in
parallel; it changes no arithmetic).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvq_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkvq_oracle.so")

BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
              "-ffp-contract=off", "-fno-strict-aliasing", "-Wall"]


def compile_to(src: str, out: str) -> str:
    """Compile one oracle source file into a shared library at `out`."""
    tmp = out + f".tmp{os.getpid()}"
    cc = os.environ.get("CC", "gcc")
    res = None
    for extra in (["-fopenmp"], []):
        cmd = [cc, *BASE_FLAGS, *extra, src, "-o", tmp, "-lm"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode == 0:
            os.replace(tmp, out)
            return out
    raise RuntimeError("oracle build failed:\n" + res.stderr)


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its source; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    return compile_to(SRC, LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
