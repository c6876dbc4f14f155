"""Build of libzyfa.so with nvcc for sm_103a (in-tree, no cmake)."""
from __future__ import annotations

import os
import shutil
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzyfa.so")
SOURCES = [os.path.join(_HERE, "csrc", f) for f in ("zyfa_api.cu", "quant.cu", "merge.cu", "host.cu")]
DEPENDS = SOURCES + [os.path.join(_HERE, "csrc", f) for f in ("fwd.cuh", "fwd3.cuh", "fwd4.cuh", "ptx.cuh")] + [
    os.path.join(os.path.dirname(_HERE), "include", "zyfa.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library (cross-compiles without a GPU)."""
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in SOURCES:                       # one nvcc per translation unit, in parallel
        obj = os.path.splitext(src)[0] + f".{os.getpid()}.o"
        cmd = [_nvcc(), ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
               "-c", "-o", obj, src]
        if verbose:
            cmd.insert(2, "-Xptxas=-v")
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    failed = [p.args for p in procs if p.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        subprocess.run([_nvcc(), ARCH, "-shared", "-o", tmp] + objs, check=True)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
