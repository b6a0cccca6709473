"""Builds the C oracle (``libssd_ref.so``) with gcc.  Test infrastructure only."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "ssd_ref.c"), os.path.join(HERE, "selective_ref.c")]
LIB = os.path.join(HERE, "libssd_ref.so")


def build(force: bool = False) -> str:
    """Compile the oracle's C files into libssd_ref.so next to them; returns the library path.

    Plain -O2 with OpenMP; no -march/-ffast-math so results are the same on
    x86_64 and aarch64 hosts (IEEE double, no reassociation).
    """
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(map(os.path.getmtime, SRCS)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-std=c11", *SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
