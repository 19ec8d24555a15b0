"""In-tree build of the C-ABI library libmoe_fp8.so for sm_103a.

Each CUDA source compiles to an object in parallel (nvcc, one -gencode), then one shared library is
linked next to this file under _lib/.  No cmake; a full build takes well under a minute.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
LIBNAME = "libmoe_fp8.so"
LIBPATH = os.path.join(LIBDIR, LIBNAME)
BUILD_DIR = os.path.join(os.path.dirname(PKG), "_build")

SOURCES = ["moe_api.cu", "moe_align.cu", "moe_quant.cu", "moe_gemm.cu", "moe_gemm_bs.cu",
           "moe_gemm_small.cu", "moe_static.cu", "moe_diag.cu"]
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-fmad=false",          # no silent multiply-add contraction: roundings are stated per step
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_fp8.so")


def _stale() -> bool:
    if not os.path.exists(LIBPATH):
        return True
    lib_mtime = os.path.getmtime(LIBPATH)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(PKG), "include", "moe_fp8.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > lib_mtime for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if it is missing or older than its sources; returns its path."""
    if not force and not _stale():
        return LIBPATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    exe = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [exe, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose:
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as pool:
        objs = list(pool.map(compile_one, SOURCES))
    tmp = LIBPATH + ".tmp"
    cmd = [exe, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIBPATH)
    return LIBPATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
