"""Build libdfl.so in-tree with nvcc for sm_103a (no CMake, parallel objects)."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libdfl.so")
# The bounds-checked variant (-DDFL_CHECK): kernels check the indices they
# compute for global accesses against the extents their shapes give, record
# DFL_ERR_BOUNDS and skip the access.  For tests; slower.
CHECK_DIR = os.path.join(OUT_DIR, "check")
LIB_CHECK = os.path.join(CHECK_DIR, "libdfl_check.so")
SOURCES = ["api.cu", "mix_rmsnorm.cu", "gemm_tc.cu", "block_attn.cu", "block_attn_tc.cu", "small_kernels.cu", "self_select.cu",
           "accept_ext.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdfl")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dfl.h"), __file__]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile every CUDA source and link libdfl.so (or, with `checked`, the
    bounds-checked libdfl_check.so); returns its path."""
    lib, out_dir = (LIB_CHECK, CHECK_DIR) if checked else (LIB, OUT_DIR)
    flags = FLAGS + (["-DDFL_CHECK"] if checked else [])
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
