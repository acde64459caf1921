"""Builds libnorm.so in-tree (``_build/``) with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically.  Rebuilds only what changed.
Run as ``python -m normalization_layernorm_rmsnorm_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures
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
LIB = os.path.join(BUILD, "libnorm.so")

SOURCES = ["api.cu", "noalloc.cu", "dropout.cu",
           "rownorm_f32.cu", "rownorm_f16.cu", "rownorm_bf16.cu",
           "batchnorm_f32.cu", "batchnorm_f16.cu", "batchnorm_bf16.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [*ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile every CUDA source and link libnorm.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    dep = _deps_mtime()
    if not force and not verbose_ptxas and os.path.exists(LIB) and os.path.getmtime(LIB) >= dep:
        return LIB
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as pool:
        objs = list(pool.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def source_digest(files=None) -> str:
    """sha256 of CUDA sources and the public header (names the kernel version
    an ncu capture was taken on): all of them, or the named files of csrc/
    (and "libnorm.h") that one kernel family is built from."""
    import hashlib
    h = hashlib.sha256()
    if files is None:
        files = sorted(glob.glob(os.path.join(CSRC, "*"))) + [os.path.join(INCLUDE, "libnorm.h")]
    else:
        files = [os.path.join(INCLUDE if f == "libnorm.h" else CSRC, f) for f in sorted(files)]
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--ptxas-v" in sys.argv))
