"""Builds libquail.so in-tree for sm_103a: nvcc for the CUDA translation units,
g++ for the host-only trie builder, compiled in parallel, linked against the
shared CUDA runtime (the one PyTorch already has loaded)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libquail.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

CUDA_SOURCES = ["api.cu", "gemm.cu", "attention.cu", "attention_tc.cu", "layer.cu", "mlp.cu", "shortlist.cu"]
CXX_SOURCES = ["trie.cpp", "cost.cpp", "shortlist.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs() -> list:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "quail.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    cuda_home = os.path.dirname(os.path.dirname(nvcc))
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        jobs.append([nvcc, *ARCH, *common, "-lineinfo", "-Xcompiler", "-fPIC", "-c",
                     os.path.join(CSRC, src), "-o", obj])
    for src in CXX_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        jobs.append([os.environ.get("CXX", "g++"), *common, "-fPIC", "-Wall", "-c",
                     "-I", os.path.join(cuda_home, "include"), os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)

    with cf.ThreadPoolExecutor(len(jobs)) as ex:
        list(ex.map(run, jobs))
    objs = [os.path.join(OUT_DIR, s + ".o") for s in CUDA_SOURCES + CXX_SOURCES]
    tmp = LIB + ".tmp"
    run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
