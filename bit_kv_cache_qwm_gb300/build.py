"""Compile libqwm (the CUDA kernels and the C ABI) for sm_103a, in-tree.

Each translation unit under csrc/ is compiled by nvcc in parallel, then the
objects are linked into bit_kv_cache_qwm_gb300/libqwm.so.  The library links
the CUDA runtime statically and depends on nothing from PyTorch.

build(debug_bounds=True) makes the checking variant libqwm_dbg.so instead
(-DQWM_DEBUG_BOUNDS: device-side checks of the centroid indices read from the
cache, which set a status bit rather than trap); the binding loads it when
QWM_DEBUG_BOUNDS=1 is set in the environment.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libqwm.so")
LIB_DBG = os.path.join(PKG, "libqwm_dbg.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqwm")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, force: bool = False, debug_bounds: bool = False) -> str:
    nvcc = _nvcc()
    out_dir = os.path.join(BUILD, "dbg") if debug_bounds else BUILD
    lib_path = LIB_DBG if debug_bounds else LIB
    os.makedirs(out_dir, exist_ok=True)
    srcs = sources()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "qwm.h"))
    newest_hdr = max(os.path.getmtime(h) for h in headers)
    flags = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
             "--expt-relaxed-constexpr"]
    if verbose:
        flags += ["-Xptxas", "-v"]
    if debug_bounds:
        flags += ["-DQWM_DEBUG_BOUNDS"]

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        if (not force and os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src)
                and os.path.getmtime(obj) >= newest_hdr):
            return obj
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    if (force or not os.path.exists(lib_path)
            or max(os.path.getmtime(o) for o in objs) > os.path.getmtime(lib_path)):
        tmp = lib_path + ".tmp"
        cmd = [nvcc, ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
