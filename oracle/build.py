"""Compile the fp64 CPU oracle (test infrastructure) into oracle/libspec_oracle.so.

Plain gcc, C11, OpenMP; no CUDA, no shared code with the product library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spec_oracle.c")
LIB = os.path.join(HERE, "libspec_oracle.so")


def build(src=SRC, out=LIB, extra_flags=(), force=False):
    """Build the oracle library; skip when it is newer than its source."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
