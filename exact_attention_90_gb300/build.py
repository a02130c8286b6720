"""Builds libfa.so in-tree with nvcc for sm_103a (no torch, no cmake).

The translation units compile in parallel (one nvcc per file) and are linked
into ``exact_attention_90_gb300/libfa.so`` with the CUDA runtime linked
statically, so the library loads on a machine without a GPU driver (the
driver is only needed once a CUDA call is made).

    python -m exact_attention_90_gb300.build [--verbose]
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
SOURCES = ["fa_api.cu", "fa_tc.cu", "fa_simt.cu", "fa_unit.cu", "fa_static.cu", "fa_bwd_simt.cu",
           "fa_bwd_tc.cu", "fa_mask.cu", "fa_host.cu"]
HEADERS = ["ptx.cuh", "tc_layout.cuh", "wait.cuh", "row_store.cuh", "fa_internal.h", "simt_tiles.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or add the CUDA toolkit to PATH)")


def _flags(extra=()):
    # FA_NVCC_FLAGS: extra nvcc flags, e.g. -D settings of the kernels' tuning
    # macros for a comparison build
    env = os.environ.get("FA_NVCC_FLAGS", "").split()
    return (ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                    "--expt-relaxed-constexpr", "-I", os.path.join(PKG, "..", "include")]
            + env + list(extra))


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files += [os.path.join(PKG, "..", "include", f) for f in ("fa.h", "fa_unit.h")]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime()


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link libfa.so; returns its path.  Raises on any failure."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc] + _flags(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = []
    for src, obj, r in results:
        if verbose or ptxas_info or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} (exit {r.returncode})")
        objs.append(obj)
    tmp = LIB + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link of libfa.so failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers/spills (-Xptxas -v)")
    ap.add_argument("--force", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force or a.ptxas_info, verbose=a.verbose, ptxas_info=a.ptxas_info))
