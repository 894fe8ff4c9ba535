"""Build step for the synthetic input generator (libsynth.so, plain C, host only)."""

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libsynth.so")


def command():
    return ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-pthread",
            os.path.join(HERE, "gen.c"), "-o", LIB]


def build():
    subprocess.run(command(), check=True)
    return LIB


if __name__ == "__main__":
    print(build())
