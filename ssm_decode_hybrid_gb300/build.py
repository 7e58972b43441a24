"""Build libreplayssm.so in-tree for sm_103a with nvcc.

Each .cu file under csrc/ is compiled to an object in parallel, then the
objects are linked into ``ssm_decode_hybrid_gb300/libreplayssm.so`` (CUDA
runtime linked statically).  Run ``python -m ssm_decode_hybrid_gb300.build``.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libreplayssm.so")
# the bounds-checked variant (-DRSSM_CHECKED: index checks that set
# RSSM_EBIT_BOUNDS instead of touching memory outside the caller's arrays)
CHECKED_BUILD = os.path.join(PKG, "_build_checked")
CHECKED_LIB = os.path.join(PKG, "libreplayssm_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose: bool = False, extra: list[str] | None = None, checked: bool = False) -> str:
    """Compile every .cu file and link the library; checked=True builds the
    bounds-checked variant (CHECKED_LIB) instead."""
    build_dir, lib = (CHECKED_BUILD, CHECKED_LIB) if checked else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    extra = list(extra or []) + (["-DRSSM_CHECKED"] if checked else [])
    srcs = sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(f"built {lib}")
    return lib


if __name__ == "__main__":
    args = sys.argv[1:]
    build(verbose=True, extra=[a for a in args if a != "--checked"], checked="--checked" in args)
