"""Compile libmoefp4.so in-tree for sm_103a with nvcc.

Each .cu under csrc/ is compiled to an object under _build/ in parallel, then
linked into block_scaled_fp4_router_gb300/libmoefp4.so (static CUDA runtime).
An up-to-date library is left alone unless force=True.

build(checked=True) makes the checked variant, libmoefp4_checked.so
(MOEFP4_CHECKED=1: caller-given indices that are out of range are recorded as
MOE_ERR_INVALID_ARG in the workspace status word), from objects under
_build/checked/.  build(trace=True) makes libmoefp4_trace.so (MOEFP4_TRACE=1:
the single-launch decode stamps %globaltimer at its phase boundaries, read
back by moe_debug_decode_trace), from objects under _build/trace/.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoefp4.so")
LIB_CHECKED = os.path.join(PKG, "libmoefp4_checked.so")
LIB_TRACE = os.path.join(PKG, "libmoefp4_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoefp4")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False, trace: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB_TRACE if trace else LIB
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    objdir = os.path.join(BUILD, "checked") if checked else os.path.join(BUILD, "trace") if trace else BUILD
    os.makedirs(objdir, exist_ok=True)
    defs = ["-DMOEFP4_CHECKED=1"] if checked else ["-DMOEFP4_TRACE=1"] if trace else []

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defs, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as pool:
        objs = list(pool.map(compile_one, _sources()))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
