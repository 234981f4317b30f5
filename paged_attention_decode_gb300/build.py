"""Build libpa_v2.so in-tree: the sm_103a kernels and the host plan behind include/pa_v2.h.

Each translation unit is compiled by nvcc in parallel for ``sm_103a`` only, then
linked into one shared library with the CUDA runtime linked statically, so the
library loads on a machine without a GPU driver (the plan and the symbol table
stay usable there; device calls then return PA_ECUDA).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libpa_v2.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
BUILD_DIR = os.path.join(ROOT, "_build")

SOURCES = ["pa_plan.cpp", "pa_cascade.cpp", "pa_partial.cu", "pa_partial_simt.cu", "pa_partial_tc.cu",
           "pa_partial_tc_cascade.cu", "pa_merge.cu", "pa_noalloc.cu", "pa_select.cu", "pa_host_step.cpp", "pa_partial_extra.cu",
           "pa_partial_extra_tc.cu", "pa_partial_extra_tc05.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libpa_v2.so")


def _compile(src: str, nvcc: str) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", f"-I{INCLUDE}",
           "-Xptxas", "-warn-spills", "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pa_v2.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False) -> str:
    """Compile and link libpa_v2.so next to this file; returns its path."""
    if not force and not _stale():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, nvcc), SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-Xlinker", "--no-undefined", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True))
