"""Compile libmuon.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each translation unit is compiled by its own nvcc process in parallel, then
linked into ``_lib/libmuon.so`` next to this file with the CUDA runtime linked
statically.  ``build(checked=True)`` makes ``_lib/libmuon_checked.so`` from the
same sources with ``-DMUON_DEVICE_CHECKS``: the kernels then test, before each
access that would fault if it broke, the invariants they rely on, and report a
broken one as MUON_ERR_DEVICE instead of making the access.  A rebuild is
skipped when the library is newer than every source and header.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libmuon.so")
LIB_CHECKED = os.path.join(OUT_DIR, "libmuon_checked.so")
SOURCES = ["api.cu", "elementwise.cu", "gemm_tc.cu", "gemm_f32.cu", "ns_static.cu", "host_stream.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(checked: bool = False) -> bool:
    lib = LIB_CHECKED if checked else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Build libmuon.so (or, checked, libmuon_checked.so) if needed and return its path."""
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(checked):
        return lib
    nvcc = _nvcc()
    obj_dir = os.path.join(OUT_DIR, "obj_checked" if checked else "obj")
    os.makedirs(obj_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else []
    if checked:
        extra.append("-DMUON_DEVICE_CHECKS")

    def compile_one(src):
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list[str]:
    """Both libraries, their translation units compiled side by side."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=2) as ex:
        return list(ex.map(lambda c: build(force=force, checked=c), (False, True)))


if __name__ == "__main__":
    if "--all" in sys.argv:
        print(build_all(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
