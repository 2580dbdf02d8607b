"""Builds libgdn.so in-tree: nvcc for sm_103a, one object per source, in parallel.

The library is written for GB300 (sm_103a) only.  Output:
``gated_delta_rule_44_gb300/_build/libgdn.so`` (git-ignored).
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libgdn.so")

SOURCES = ["gdn_api.cpp", "gdn_status.cu", "gdn_prepare.cu", "gdn_recurrent.cu", "gdn_fused.cu",
           "gdn_chunked.cu", "gdn_kda_chunked.cu", "gdn_noalloc.cu", "gdn_norm.cu", "gdn_packed.cu"]
HEADERS = ["gdn_internal.h", "tcgen05.cuh", "gdn_math.cuh", "gdn_rowstep.cuh", "gdn_chunk_common.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the GDN CUDA library cannot be built")


def _fingerprint() -> str:
    h = hashlib.sha256()
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(INCLUDE, "gdn.h")]
    for f in files:
        if os.path.exists(f):
            with open(f, "rb") as fh:
                h.update(fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def _compile(src: str, extra: List[str]) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def build_library(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile (if stale) and return the path of libgdn.so."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "libgdn.stamp")
    fp = _fingerprint()
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as fh:
            if fh.read().strip() == fp:
                return LIB
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "--cudart", "shared", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(fp)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True))
