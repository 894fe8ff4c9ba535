"""Build step for the synthetic input generator: libsynth.so (plain C, host)
and libsynth_dev.so (the same definition on the GPU, nvcc for sm_103a)."""

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libsynth.so")
DEV_LIB = os.path.join(HERE, "libsynth_dev.so")


def command():
    return ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-pthread",
            os.path.join(HERE, "gen.c"), "-o", LIB]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def dev_command():
    return [nvcc(), "-O3", "-shared", "-Xcompiler", "-fPIC", "-gencode", "arch=compute_103a,code=sm_103a",
            "-lineinfo", "-fmad=false", "-cudart", "shared", os.path.join(HERE, "gen_dev.cu"), "-o",
            DEV_LIB + ".tmp"]


def build():
    dev = subprocess.Popen(dev_command(), stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    subprocess.run(command(), check=True)
    out, _ = dev.communicate()
    if dev.returncode != 0:
        raise RuntimeError("nvcc failed for gen_dev.cu:\n" + out)
    os.replace(DEV_LIB + ".tmp", DEV_LIB)
    return LIB


if __name__ == "__main__":
    print(build())
