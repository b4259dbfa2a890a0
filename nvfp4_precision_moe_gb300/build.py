"""Builds the CUDA library libnvfp4moe.so for sm_103a with nvcc.

Each .cu file is compiled in parallel (one -gencode, compute_103a/sm_103a),
then linked into a shared library in ``_build/`` next to this file.  The
CUDA runtime is linked statically; the driver entry point for TMA descriptors
is looked up at run time, so the library has no libcuda link dependency.
"""
import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libnvfp4moe.so")
SOURCES = ["abi.cu", "quantize.cu", "moe.cu", "gemm.cu", "gemm_single.cu", "gemm_pair.cu", "train.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def _nvcc():
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the NVFP4 CUDA library cannot be built")
    return p


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, "common.cuh"),
                                                        os.path.join(CSRC, "gemm_common.cuh"),
                                                        os.path.join(INCLUDE, "nvfp4moe.h")]
    return files


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources (if stale) and return the path of the .so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(f) for f in _inputs())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s" % (src, r.stderr))
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n%s" % r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
