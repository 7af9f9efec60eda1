"""Build libnmmlp.so (the C-ABI library) in-tree with nvcc for sm_103a.

Usage: python -m mlp_neural_gb300.build [--force] [--checked]
Objects go to _build/ at the repository root; the library is written to
mlp_neural_gb300/libnmmlp.so. The CUDA runtime is linked statically, so the
library loads on a machine without a GPU driver (calls then fail with
NM_ERR_CUDA instead of the library failing to load).

--checked builds the checking library instead, libnmmlp_check.so (objects in
_build/check/): the same sources with NM_RANGE_CHECKS defined, whose kernels
check every tensor- and shared-memory range they touch against the plan and
report a miss as NM_ERR_RANGE_CHECK.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libnmmlp.so")
LIB_CHECK = os.path.join(PKG, "libnmmlp_check.so")

SOURCES = ["nm_api.cu", "nm_fused.cu", "nm_noalloc.cu"]
HEADERS = ["nm_internal.h", "nm_layout.cuh", "nm_ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "nm_mlp.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(checked: bool = False) -> bool:
    lib = LIB_CHECK if checked else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECK if checked else LIB
    if not force and up_to_date(checked):
        return lib
    out_dir = os.path.join(BUILD, "check") if checked else BUILD
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + (["-DNM_RANGE_CHECKS"] if checked else [])

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))
