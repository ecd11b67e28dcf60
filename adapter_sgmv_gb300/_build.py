"""Compile the CUDA library ``liblora_sgmv.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in parallel with nvcc, then the
objects are linked into one shared library next to this file.  ``debug=True``
builds ``liblora_sgmv_debug.so`` instead: the same sources and ABI with
LORA_DEBUG_CHECKS=1, which compiles in the device-side checks of every index
read from the routing metadata (an index out of range sets LORA_ERR_INDEX in
the status word and is redirected in range; nothing traps).  The CUDA
runtime is linked statically; the driver API is reached through the
runtime's entry-point query, so the library loads on a machine without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "liblora_sgmv.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
DEBUG_LIB_PATH = os.path.join(PKG, "liblora_sgmv_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblora_sgmv.so")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, debug: bool = False) -> str:
    """Build (if needed) and return the path of ``liblora_sgmv.so`` (``debug``:
    of ``liblora_sgmv_debug.so``, with the device-side index checks)."""
    build_dir = os.path.join(BUILD_DIR, "debug") if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    exe = nvcc()
    flags = list(NVCC_FLAGS)
    if debug:
        flags += ["-DLORA_DEBUG_CHECKS=1"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        if not force and not _stale(obj, [src] + hdrs):
            return obj, ""
        cmd = [exe, *ARCH, *flags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stdout + res.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, max(1, len(srcs)))) as ex:
        results = list(ex.map(compile_one, srcs))
    objs = [o for o, _ in results]
    if verbose or ptxas_verbose:
        for o, log in results:
            if log:
                print(f"== {os.path.basename(o)}\n{log}")
    if force or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [exe, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
