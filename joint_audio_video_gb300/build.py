"""Build libh3attn.so in-tree for sm_103a with nvcc (no CMake, no torch extension).

Each translation unit is compiled in parallel into ``_obj/``; the shared
library links the CUDA runtime statically, so it has no load-time dependency
on a GPU driver.  A source newer than the library (or a changed flag set)
triggers a rebuild.  ``build(checked=True)`` builds the checked library
(``libh3attn_checked.so`` from ``_obj_checked/``, compiled with H3_CHECKED:
every global access a kernel addresses itself is tested against its buffer's
extents first).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_obj")
LIB = os.path.join(PKG, "libh3attn.so")
OBJ_CHECKED = os.path.join(PKG, "_obj_checked")
LIB_CHECKED = os.path.join(PKG, "libh3attn_checked.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
           "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]
SOURCES = ["h3attn_api.cu", "adaln.cu", "mrope.cu", "gemm.cu", "attn.cu", "layout.cpp",
           "noalloc.cu", "denoise.cu", "quant.cu"]
HEADERS = ["ptx.cuh", "tmap.hpp", "kernels.hpp"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the h3attn CUDA library cannot be built")


def _stamp(flags) -> str:
    h = hashlib.sha256()
    h.update(" ".join(ARCH + flags).encode())
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    with open(os.path.join(INCLUDE, "h3attn.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def _compile(src: str, verbose: bool, obj_dir: str, flags) -> str:
    obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    with open(os.path.join(obj_dir, os.path.splitext(src)[0] + ".ptxas.txt"), "w") as f:
        f.write(r.stderr)
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile the library (or, with ``checked``, the checked library) if it is
    missing or stale; return its path."""
    obj_dir, lib = (OBJ_CHECKED, LIB_CHECKED) if checked else (OBJ, LIB)
    flags = CUFLAGS + (["-DH3_CHECKED"] if checked else [])
    os.makedirs(obj_dir, exist_ok=True)
    stamp_file = os.path.join(obj_dir, "stamp")
    stamp = _stamp(flags)
    if not force and os.path.exists(lib) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return lib
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, obj_dir, flags), SOURCES))
    tmp = lib + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))
