"""Builds the in-tree CUDA library ``_lib/libkpooldsa.so`` for sm_103a.

Each ``csrc/*.cu`` file is compiled by nvcc in parallel (skipped when its
object is newer than every source and header), then linked into one shared
library with the C ABI of ``include/kpooldsa.h``.

``build(checked=True)`` builds the same sources with ``-DKPOOL_CHECKED`` into
``_lib/libkpooldsa_checked.so``: internal bounds checks on the indexer's
computed indices then record ``KPOOL_ERR_CHECK`` in the status word instead of
being compiled out (a stand-in for a memory checker, which this pool does not
offer).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libkpooldsa.so")
OBJDIR_CHECKED = os.path.join(LIBDIR, "obj_checked")
LIB_CHECKED = os.path.join(LIBDIR, "libkpooldsa_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return max(os.path.getmtime(f) for f in files)


def build(verbose: bool = False, force: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile and link; returns the library path.  Raises on a compiler error."""
    objdir, lib = (OBJDIR_CHECKED, LIB_CHECKED) if checked else (OBJDIR, LIB)
    if checked:
        extra_flags = (*extra_flags, "-DKPOOL_CHECKED")
    os.makedirs(objdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest = _deps_mtime()
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        if not force and os.path.exists(obj) and os.path.getmtime(obj) >= newest:
            return obj
        cmd = [cc, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        cmd = [cc, *ARCH, "-shared", "-o", lib, *objs, "-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    import sys
    print(build(verbose=True, force="--force" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ()))
