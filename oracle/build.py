"""Compile the C oracle into oracle/liboracle_nvfp4.so.

Test infrastructure: the oracle is the checker for the CUDA library and is never linked into it.
The flags keep every float operation a single IEEE-754 binary32 operation: no contraction of
a*b+c into fused multiply-adds and no fast-math.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "nvfp4_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle_nvfp4.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-Werror"]


def command():
    return ["gcc", *CFLAGS, SOURCE, "-o", LIBRARY, "-lm"]


def build(force=False):
    """Build the oracle library if it is missing or older than its source; return its path."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    subprocess.run(command(), check=True)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
