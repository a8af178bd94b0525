"""Build step for the CPU oracle (test infrastructure only).

Compiles ``gemm_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc and
OpenMP. Floating-point contraction is switched off so that the file means the
same thing on x86-64 and AArch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "gemm_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "liboracle.so")

CFLAGS = ["-O3", "-std=c11", "-fPIC", "-shared", "-fopenmp",
          "-ffp-contract=off", "-fno-fast-math"]


def compile_oracle(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile ``source`` into the shared library ``output``; return its path."""
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = output + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


def ensure_built() -> str:
    """Build the oracle if the library is missing or older than its source."""
    if (not os.path.exists(LIBRARY)
            or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
        compile_oracle()
    return LIBRARY


if __name__ == "__main__":
    print(compile_oracle(*sys.argv[1:3]))
