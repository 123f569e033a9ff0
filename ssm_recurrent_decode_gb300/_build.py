"""Builds libgdn_decode.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit is compiled in parallel to an object file, then the objects are linked
into ``ssm_recurrent_decode_gb300/_lib/libgdn_decode.so``. A rebuild happens only when a source or
header is newer than the library. No GPU is needed to build.

``build(debug=True)`` makes ``libgdn_decode_debug.so`` from the same sources with ``-DGDN_DEBUG``:
its kernels check the indices they compute and report one outside its range through the error
word (GDN_DEVERR_RANGE) instead of making the access. It is for tests, not for timing.
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
LIBPATH = os.path.join(LIBDIR, "libgdn_decode.so")
DEBUG_LIBPATH = os.path.join(LIBDIR, "libgdn_decode_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
              "-fno-strict-aliasing", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libgdn_decode.so")
    return exe


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(debug: bool = False) -> bool:
    path = DEBUG_LIBPATH if debug else LIBPATH
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link the library (the debug variant with debug=True) if needed; returns its
    path."""
    libpath = DEBUG_LIBPATH if debug else LIBPATH
    if not force and up_to_date(debug):
        return libpath
    objdir = os.path.join(LIBDIR, "obj_debug" if debug else "obj")
    os.makedirs(objdir, exist_ok=True)
    exe = nvcc()
    extra = ["-DGDN_DEBUG"] if debug else []

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = f"{libpath}.{os.getpid()}.tmp"
    r = subprocess.run([exe, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"linking {os.path.basename(libpath)} failed:\n{r.stderr}")
    os.replace(tmp, libpath)
    return libpath


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
