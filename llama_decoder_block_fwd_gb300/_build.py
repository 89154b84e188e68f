"""Build the in-tree CUDA library (libllama_block.so) for sm_103a with nvcc.

Each .cu file compiles to an object in parallel, then nvcc links them into one shared
library with the CUDA runtime linked statically, so the library has no link-time
dependency on libcuda (the driver is reached through the runtime's entry-point query).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libllama_block.so")
# the bounds-checking build (-DLLAMA_DEBUG): same sources, its own objects and library
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libllama_block_debug.so")
SOURCES = ["api.cu", "kernels_simt.cu", "gemm_tc.cu", "gemm_tc2.cu", "gemm_skinny.cu", "attn_tc.cu", "decode_attn.cu", "decode_fin.cu", "sample.cu", "decode_attn8.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, build_dir: str, extra: tuple) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, debug: bool = False) -> str:
    """Build libllama_block.so, or with debug=True the bounds-checking libllama_block_debug.so."""
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    extra = ("-DLLAMA_DEBUG",) if debug else ()
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda src: _compile(src, build_dir, extra), SOURCES))
    objs = [o for o, _ in results]
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        for (o, log), src in zip(results, SOURCES):
            f.write(f"== {src}\n{log}\n")
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(open(os.path.join(build_dir, "ptxas.log")).read())
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, debug="--debug" in sys.argv))
