"""Builds libdsaprep.so in-tree with nvcc for sm_103a (no torch extension
machinery: the library is plain C ABI over CUDA)."""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libdsaprep.so")
INCLUDE = os.path.join(ROOT, "include")
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "--diag-suppress=177",
    "-Xcompiler", "-fPIC", "-shared",
    "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(PKG, "csrc", "*.cu")))


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    deps = sources() + glob.glob(os.path.join(PKG, "csrc", "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu under csrc/ (in parallel, one nvcc per file) and
    link them into one shared library."""
    if not force and not _stale():
        return LIB_PATH
    tag = f"{os.getpid()}"
    objs, procs = [], []
    compile_flags = [f for f in NVCC_FLAGS if f not in ("-shared",)]
    for src in sources():
        obj = os.path.join(PKG, "csrc", os.path.basename(src) + f".{tag}.o")
        cmd = [_nvcc(), *compile_flags, "-I", INCLUDE, "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append(subprocess.Popen(cmd))
        objs.append(obj)
    try:
        codes = [p.wait() for p in procs]
        if any(codes):
            raise subprocess.CalledProcessError(max(codes), "nvcc -c")
        tmp = LIB_PATH + f".tmp{tag}"
        subprocess.check_call([_nvcc(), *NVCC_FLAGS, "-o", tmp, *objs])
        os.replace(tmp, LIB_PATH)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB_PATH
