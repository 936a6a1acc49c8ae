"""Compile the CUDA library (libspecv.so) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libspecv.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecv")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(d) > os.path.getmtime(out) for d in deps)


def build(force: bool = False, verbose: bool = False, out: str = LIB) -> str:
    """Each translation unit compiled to an object in parallel (one per kernel
    mode), then linked into the shared library."""
    if not force and not _stale(out):
        return out
    nvcc = _nvcc()
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    objdir = os.path.join(PKG, "_build")
    os.makedirs(objdir, exist_ok=True)
    common = [nvcc, ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE]
    if verbose:
        common.insert(1, "-Xptxas=-v")
    procs = []
    for src in sources():
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        procs.append((src, obj, subprocess.Popen(common + ["-c", src, "-o", obj],
                                                 stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                                 text=True)))
    logs, failed = [], []
    for src, obj, p in procs:
        o, e = p.communicate()
        logs.append(o + e)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed on " + ", ".join(failed) + ":\n" + "".join(logs))
    link = [nvcc, ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath," + cuda_lib,
            "-o", out + ".tmp"] + [obj for _, obj, _ in procs]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
    os.replace(out + ".tmp", out)
    if verbose:
        print("".join(logs))
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
