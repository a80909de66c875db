"""Build the package's CUDA libraries in-tree with nvcc for sm_103a.

    python -m selective_state_space_140_b300.build [--force] [--ptxas-info]

libmamba_scan.so   <- csrc/*.cu          (the scan's C ABI, include/mamba_scan.h)
libmamba_ubench.so <- csrc/ubench/*.cu   (roofline micro-benchmarks, include/mamba_ubench.h)

Every .cu file is compiled separately (in parallel) and linked into its
library.  A library is rebuilt only when a source or header is newer.
"""
from __future__ import annotations

import argparse
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmamba_scan.so")
UBENCH_LIB = os.path.join(PKG, "libmamba_ubench.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def sources(lib: str = LIB):
    sub = CSRC if lib == LIB else os.path.join(CSRC, "ubench")
    return sorted(glob.glob(os.path.join(sub, "*.cu")))


def _deps(lib: str):
    return sources(lib) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps(lib))


def _compile(src: str, ptxas_info: bool) -> tuple[str, str]:
    rel = os.path.relpath(src, CSRC).replace(os.sep, "_")
    obj = os.path.join(OBJ, rel + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
    if ptxas_info:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _build_one(lib: str, force: bool, ptxas_info: bool, quiet: bool) -> str:
    if not force and not ptxas_info and up_to_date(lib):
        return lib
    os.makedirs(OBJ, exist_ok=True)
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_info), sources(lib)))
    if ptxas_info or not quiet:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib + ".tmp"
    # --no-undefined: a missing definition fails here, not when the library loads
    cmd = [NVCC, *ARCH, "-shared", "-Xlinker", "--no-undefined", "-o", tmp,
           *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, ptxas_info: bool = False, quiet: bool = True) -> str:
    """Compile and link both libraries; return the scan library's path."""
    _build_one(UBENCH_LIB, force, ptxas_info, quiet)
    return _build_one(LIB, force, ptxas_info, quiet)


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, ptxas_info=args.ptxas_info, quiet=False))
