"""Build libkda.so in-tree with nvcc for sm_103a.

Each .cu under csrc/ is compiled to an object in parallel, then linked into
``gated_delta_rule_intra_gb300/libkda.so`` (git-ignored).  No CMake, no torch
extension machinery: the library is a plain C-ABI shared object.
``build_debug_library()`` builds the same sources with ``-DKDA_DEBUG_CHECKS`` into
``libkda_debug.so``: every global index the kernels compute is checked against its
buffer's extent and reported through ``kda_debug_set_flags`` (tests only).
"""

from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libkda.so")
DEBUG_LIB = os.path.join(PKG, "libkda_debug.so")
BUILD_DIR = os.path.join(PKG, "_build")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Hidden visibility: only the C ABI (kda_api.cu) is exported.  Two builds loaded in one
# process (libkda.so and libkda_debug.so) then share no C++ internals; in particular no
# function-local static of a template becomes a process-wide unique symbol.
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkda")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _compile(src: str, extra, build_dir: str) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def build_library(out: str = LIB, extra_flags=(), verbose: bool = False,
                  build_dir: str = BUILD_DIR) -> str:
    """Compile every csrc/*.cu for sm_103a and link libkda.so; returns its path."""
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra_flags), build_dir), srcs))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(f"built {out}")
    return out


def build_debug_library(verbose: bool = False) -> str:
    """The bounds-checked debug build, libkda_debug.so; returns its path."""
    return build_library(DEBUG_LIB, ["-DKDA_DEBUG_CHECKS"], verbose, DEBUG_BUILD_DIR)


if __name__ == "__main__":
    build_library(verbose=True)
    build_debug_library(verbose=True)
