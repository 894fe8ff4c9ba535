"""Build step for liblst.so: nvcc for sm_103a, in-tree, translation units in parallel."""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "liblst.so")

SOURCES = ["lst_layout.cpp", "lst_api.cpp", "lst_stream.cpp", "lst_store.cpp", "lst_kernels.cu", "lst_kernels_ex.cu", "lst_noalloc.cu", "lst_copy.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def compile_cmd(src: str, obj: str) -> list:
    cmd = [nvcc(), "-c", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
           "-I", os.path.join(ROOT, "include"), "-o", obj, src]
    if src.endswith(".cu"):
        # IEEE division/sqrt and no flush-to-zero are nvcc's defaults; they are
        # spelled out because the update must match the fp32 reference exactly.
        cmd += ARCH + ["-lineinfo", "-prec-div=true", "-prec-sqrt=true", "-ftz=false", "-fmad=false",
                       "-Xptxas", "-v"]
    else:
        cmd += ["-x", "c++"]
    return cmd


def build(verbose: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    procs = []
    objs = []
    for s in SOURCES:
        obj = os.path.join(OBJ, os.path.splitext(s)[0] + ".o")
        objs.append(obj)
        cmd = compile_cmd(os.path.join(CSRC, s), obj)
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(s)
            sys.stderr.write(out)
        elif verbose and out:
            sys.stderr.write(out)
        if s.endswith(".cu") and out:
            with open(os.path.join(OBJ, "ptxas_" + os.path.splitext(s)[0] + ".txt"), "w") as f:
                f.write(out)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + ".tmp"
    subprocess.run([nvcc(), "-shared", "-o", tmp] + objs + ["-cudart", "shared", "-lpthread"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
