"""Build liblinattn.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit under ``csrc/`` is compiled in parallel, then the
objects are linked into ``_build/liblinattn.so`` against the shared CUDA
runtime (the same libcudart.so that PyTorch loads).  Run as a module
(``python -m causal_kernelized_linear_gb300.build``) or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liblinattn.so")
# the LA_DEBUG build (device-side index checks), apart from the product library
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_BUILD_DIR, "liblinattn.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
CXX_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
             "--expt-relaxed-constexpr", "-Xptxas", "-O3"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblinattn")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(debug: bool = False) -> bool:
    path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          debug: bool = False) -> str:
    """Compile every ``csrc/*.cu`` for sm_103a and link liblinattn.so; with
    ``debug``, the LA_DEBUG build (kernels check their indices) in a folder
    of its own."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and up_to_date(debug):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if debug:
        extra.append("-DLA_DEBUG")

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH_FLAGS, *CXX_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_verbose:
        for obj, log in results:
            if log.strip():
                print(f"== {os.path.basename(obj)}\n{log}", file=sys.stderr)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH_FLAGS, "-shared", "-cudart", "shared", "-o", tmp,
           *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas-v" in sys.argv,
                debug="--debug" in sys.argv))
