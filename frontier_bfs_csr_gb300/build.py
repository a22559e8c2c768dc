"""Build the CUDA library ``libbfs_csr.so`` in-tree with nvcc for sm_103a.

One translation unit (``csrc/bfs_csr.cu``), one ``-gencode``; the CUDA runtime
is linked statically. The result lands next to this file, where the Python
binding loads it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SOURCES = [os.path.join(HERE, "csrc", "bfs_csr.cu")]
DEPENDS = SOURCES + [os.path.join(HERE, "csrc", "bfs_device.cuh"),
                     os.path.join(HERE, "csrc", "walk_device.cuh"),
                     os.path.join(ROOT, "include", "bfs_csr.h")]
LIB = os.path.join(HERE, "libbfs_csr.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbfs_csr.so")
    return path


def command(out: str = LIB, verbose_ptxas: bool = False) -> list[str]:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-I", os.path.join(ROOT, "include"), "-o", out, *SOURCES]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    stale = not os.path.exists(LIB) or any(os.path.getmtime(d) > os.path.getmtime(LIB)
                                           for d in DEPENDS)
    if force or stale or verbose_ptxas:
        tmp = LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(command(tmp, verbose_ptxas))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose_ptxas="-v" in sys.argv)
    print(LIB)
