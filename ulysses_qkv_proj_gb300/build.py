"""Build libqnre.so in-tree with nvcc for sm_103a.

    python -m ulysses_qkv_proj_gb300.build            # libqnre.so
    python -m ulysses_qkv_proj_gb300.build --debug    # libqnre_debug.so: bounds-checked accesses

Compiles every csrc/*.cu in parallel, then links the shared library next to
this file.  Only nvcc and the CUDA runtime (linked statically) are needed; the
driver entry point for TMA descriptors is looked up at run time, so the library
also loads on a machine without a GPU driver.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libqnre.so")
DEBUG_BUILD_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(HERE, "libqnre_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              f"-I{INCLUDE}", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, ptxas_info: bool = False, debug_bounds: bool = False) -> str:
    """Compile and link the library; `debug_bounds` builds libqnre_debug.so, whose
    kernels check every load and store against its buffer's byte range and skip
    (and count) any access outside it."""
    nvcc = _nvcc()
    build_dir = DEBUG_BUILD_DIR if debug_bounds else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    defines = ["-DQNRE_DEBUG_BOUNDS=1"] if debug_bounds else []
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defines, "-c", src, "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose or ptxas_info:
            sys.stdout.write(res.stdout + res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv, debug_bounds="--debug" in sys.argv))
