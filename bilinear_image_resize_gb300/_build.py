"""Builds ``libgbresize.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel, then nvcc links the shared
library (CUDA runtime linked statically, so the library needs no CUDA
libraries at load time).  A rebuild happens only when a source or header is
newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build_obj")
SOURCES = ["kernels.cu", "stream.cu", "direct.cu", "filter.cu", "texture.cu", "multi.cu", "api.cu", "noalloc.cu", "baseline_copy.cu", "filter_tc.cu"]
HEADERS = [os.path.join(CSRC, "rz_internal.h"), os.path.join(CSRC, "rz_device.h"), os.path.join(INCLUDE, "gbresize.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]


# The bounds-checked variant (libgbresize_checked.so, for tests): these
# sources compile with -DRZ_CHECK_BOUNDS; the others are the normal build's
# objects.
CHECKED_SOURCES = ["kernels.cu", "stream.cu", "direct.cu", "api.cu", "noalloc.cu"]


def library_path(checked: bool = False) -> str:
    return os.path.join(PKG, "libgbresize_checked.so" if checked else "libgbresize.so")


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Build libgbresize.so (or, with checked=True, after the normal build,
    libgbresize_checked.so: the bounds-checked variant)."""
    if checked:
        build(force=force, verbose=verbose, extra_flags=extra_flags)
    os.makedirs(BUILD, exist_ok=True)
    lib = library_path(checked)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if not force and not _stale(lib, srcs + HEADERS + [os.path.abspath(__file__)]):
        return lib
    nvcc = _nvcc()

    def compile_one(src):
        name = os.path.basename(src)
        if checked and name not in CHECKED_SOURCES:
            return os.path.join(BUILD, name + ".o")    # the normal build's object
        obj = os.path.join(BUILD, name + (".checked.o" if checked else ".o"))
        flags = [*extra_flags, "-DRZ_CHECK_BOUNDS"] if checked else list(extra_flags)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
