"""Build libproj_gb300 (the C-ABI library) with nvcc for sm_103a, in-tree.

Each translation unit is compiled in parallel; the shared library lands next to
this file as ``libproj_gb300.<machine>.so`` (the machine suffix keeps x86 and
Arm builds apart).  Objects go to ``_build/<machine>/``.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = ["proj_api.cu", "planner.cpp", "kernel_tc_lean.cu", "kernel_tc_fused.cu", "kernel_tc_pair.cu",
           "kernel_tc_pair_fused.cu"]
HEADERS = [os.path.join(CSRC, "proj_internal.h"), os.path.join(CSRC, "proj_kernel.cuh"),
           os.path.join(CSRC, "proj_aux.cuh"), os.path.join(CSRC, "proj_launch.h"),
           os.path.join(INCLUDE, "proj.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libproj_gb300")


def library_path() -> str:
    return os.path.join(PKG, f"libproj_gb300.{platform.machine()}.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if sources changed) and return the library path."""
    out = library_path()
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if not force and not _stale(out, srcs + HEADERS):
        return out
    objdir = os.path.join(PKG, "_build", platform.machine())
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH_FLAGS, *COMMON, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
