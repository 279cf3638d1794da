"""Build the sm_103a CUDA library ``_build/libgb300attn.so`` in-tree with nvcc.

One translation unit (``csrc/attn_api.cu``), one ``-gencode`` (compute_103a -> sm_103a), the CUDA
runtime linked as a shared library (the same ``libcudart`` PyTorch already loaded) with an rpath to
the toolkit's lib64 for stand-alone C callers.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libgb300attn.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
# The debug build (-DATTN_DEBUG): every kernel checks the indices behind its computed stores and
# records a failed check in the device status word instead of storing (no trap).
DEBUG_LIB_PATH = os.path.join(BUILD_DIR, "libgb300attn_debug.so")
SOURCES = [os.path.join(CSRC, "attn_api.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in (
    "attn_fwd_kernel.cuh", "attn_fwd_pair_kernel.cuh", "attn_fwd_d256_kernel.cuh", "attn_bwd_kernel.cuh",
    "mla_decode_kernel.cuh", "ptx.cuh")] + [
    os.path.join(INCLUDE, "attn.h")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def nvcc_command(out_path: str, extra=()) -> list:
    home = cuda_home()
    lib64 = os.path.join(home, "lib64")
    return [os.path.join(home, "bin", "nvcc"), *ARCH_FLAGS, "-lineinfo", "-O3", "-std=c++17",
            "-Xcompiler", "-fPIC,-O2", "-shared", "-cudart", "shared", f"-I{INCLUDE}",
            f"-I{CSRC}", f"-Xlinker", f"-rpath,{lib64}", *extra, "-o", out_path, *SOURCES]


def is_fresh(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in DEPENDS)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    """Compile the library (or, with debug=True, its index-checking debug build) unless it is up
    to date; returns its path."""
    path = DEBUG_LIB_PATH if debug else LIB_PATH
    if is_fresh(path) and not force and not ptxas_info:
        return path
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = f"{path}.{os.getpid()}.tmp"
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug:
        extra.append("-DATTN_DEBUG")
    cmd = nvcc_command(tmp, extra)
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if ptxas_info or verbose:
        print(res.stdout + res.stderr, file=sys.stderr)
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
