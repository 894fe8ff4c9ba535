"""Build step for the oracle's C library (liboracle.so). Test infrastructure only."""

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "liboracle.so")


def command():
    # No contraction and no fast-math: every fp32 operation is rounded on its own.
    return ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
            os.path.join(HERE, "oracle.c"), "-lm", "-o", LIB]


def build():
    subprocess.run(command(), check=True)
    return LIB


if __name__ == "__main__":
    print(build())
