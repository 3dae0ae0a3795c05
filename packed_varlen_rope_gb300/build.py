"""Build librope_qk.so in the package directory with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SOURCES = [os.path.join(HERE, "csrc", n) for n in ("rope_qk.cu", "rope_host.cu", "glu.cu")]
HEADERS = [os.path.join(ROOT, "include", "rope_qk.h"), os.path.join(ROOT, "include", "glu.h"),
           os.path.join(HERE, "csrc", "fastdiv.cuh"), os.path.join(HERE, "csrc", "cos_sin.cuh")]
LIB_PATH = os.path.join(HERE, "librope_qk.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def flags(verbose_ptxas: bool = False):
    f = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
         "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the CUDA library if it is missing or older than its sources."""
    if force or verbose_ptxas or stale():
        tmp = LIB_PATH + ".tmp%d" % os.getpid()
        cmd = [nvcc(), *flags(verbose_ptxas), *SOURCES, "-o", tmp]
        subprocess.check_call(cmd)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force=True, verbose_ptxas="-v" in sys.argv)
    print(LIB_PATH)
