"""Compile the float64 sink-attention oracle into a shared library.

TEST INFRASTRUCTURE: the library this builds is loaded only by the tests, the
smoke check and the benchmark's CPU-baseline leg.

Plain gcc, no vendor code, no fast-math: the oracle must keep IEEE double
semantics. Run as ``python -m oracle.build`` or through ``build()``.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sinkattn_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libsinkattn_oracle.so")


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra",
           SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
