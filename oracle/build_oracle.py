"""Compile the fp64 CPU oracle (oracle/cporacle.c) into oracle/_build/libcporacle.so.

The oracle is test infrastructure: the test-suite, the smoke check and the
CPU-baseline leg of the benchmark load it; the CUDA library never does.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cporacle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libcporacle.so")


def build(force: bool = False) -> str:
    """Build the shared library if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
