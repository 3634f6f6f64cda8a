"""Compile the CPU oracle (``oracle.c``) into ``liboracle.so`` beside it.

Test infrastructure: the oracle is the checker, not part of the library. Plain
gcc, no fast-math, no contraction, OpenMP for the loop over output columns.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

FLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
         "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the shared library if it is missing or older than its source."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    tmp = LIBRARY + f".{os.getpid()}.tmp"
    cmd = ["gcc", *FLAGS, SOURCE, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
