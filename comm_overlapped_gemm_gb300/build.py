"""Build the CUDA library libtdx.so in-tree for sm_103a.

Each translation unit under csrc/ is compiled by its own nvcc process (in parallel), then linked
into comm_overlapped_gemm_gb300/_lib/libtdx.so with the CUDA runtime linked statically, so that
loading the library needs no libcudart on the library path. Run ``python
comm_overlapped_gemm_gb300/build.py`` (this file never imports the package, whose import loads the
library) or load this file by path and call :func:`build`.
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
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(LIBDIR, "libtdx.so")
SOURCES = ["tdx_api.cu", "tdx_kernel_bf16.cu", "tdx_kernel_fp8.cu", "tdx_moe.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, log_dir: str) -> str:
    obj = os.path.join(OBJDIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(log_dir, os.path.splitext(src)[0] + ".ptxas.txt"), "w") as f:
        f.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stderr[-4000:]}")
    return obj


def build(verbose: bool = False) -> str:
    """Compile every translation unit and link libtdx.so. Returns the library path."""
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(OBJDIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, OBJDIR), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr[-4000:]}")
    os.replace(tmp, LIB)
    if verbose:
        for s in SOURCES:
            with open(os.path.join(OBJDIR, os.path.splitext(s)[0] + ".ptxas.txt")) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
