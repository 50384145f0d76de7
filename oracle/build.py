"""Build the fp64 CPU oracle (``liboracle.so``) with gcc.

Test infrastructure only: the oracle is the checker, never the product path.
Plain ``-O2``, single-threaded, no OpenMP, so its timing is that of the
oracle as it stands.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it; return the library path."""
    deps = [SRC, os.path.join(HERE, "oracle.h")]
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(d) for d in deps)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
