"""Build libmslkb.so in-tree with nvcc for sm_103a (GB300).

    python -m fp8_rowwise_scaled_gb300.build [--force] [--ptxas-verbose] [--checked]

--checked builds libmslkb_checked.so instead: the same sources compiled with MSLKB_CHECKED,
whose kernels test every global access against the extents of the call's buffers and
report an index outside them in the device status word (MSLKB_DEV_BOUNDS) instead of
making the access.  A test build (the stand-in for a memory checker); slower.

Each translation unit in csrc/ compiles in parallel to _build/*.o, then nvcc links them
into fp8_rowwise_scaled_gb300/libmslkb.so (CUDA runtime linked statically; the CUDA driver's
tensor-map encoder is fetched at run time, so the library loads on a machine without a
GPU).  Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmslkb.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libmslkb_checked.so")
SOURCES = ["mslkb.cu", "mslkb_noalloc.cu", "variants_stacked_tma.cu",
           "variants_dynamic_tma.cu", "variants_cpasync.cu", "variants_ragged_n.cu",
           "variants_ragged_k.cu", "variants_blockscale.cu", "variants_blockscale_dynamic.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA 13 toolkit required to build libmslkb.so)")


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES] + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str, ptxas_verbose: bool, checked: bool = False) -> tuple[str, str]:
    obj = os.path.join(BUILD_CHECKED if checked else BUILD,
                       os.path.splitext(os.path.basename(src))[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
           "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if checked:
        cmd.insert(1, "-DMSLKB_CHECKED")
    if ptxas_verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          checked: bool = False) -> str:
    """Compile and link libmslkb.so (checked: libmslkb_checked.so); returns its path."""
    lib = LIB_CHECKED if checked else LIB
    if not force and not ptxas_verbose and up_to_date(lib):
        return lib
    os.makedirs(BUILD_CHECKED if checked else BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose, checked), srcs))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    ap.add_argument("--checked", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=True, ptxas_verbose=a.ptxas_verbose, checked=a.checked))
