"""Build libmla.so in-tree for sm_103a with nvcc (no torch extension machinery).

Each CUDA translation unit compiles in parallel; the objects are linked into
``mla_latent_cache_gb300/libmla.so`` against the shared CUDA runtime.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmla.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
           "-Xptxas", "-v", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmla.so")


def _sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cuh", ".h")):
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _compile(nvcc: str, src: str, hdr: str, verbose: bool) -> tuple[str, str]:
    with open(src, "rb") as fh:
        key = hashlib.sha256(fh.read() + hdr.encode() + " ".join(ARCH + NVFLAGS).encode()).hexdigest()[:16]
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + f".{key}.o")
    log = ""
    if not os.path.exists(obj):
        cmd = [nvcc, *ARCH, *NVFLAGS, "-c", src, "-o", obj + ".tmp"]
        p = subprocess.run(cmd, capture_output=True, text=True)
        log = p.stdout + p.stderr
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{log}")
        os.replace(obj + ".tmp", obj)
        with open(obj + ".log", "w") as fh:
            fh.write(log)
    elif verbose and os.path.exists(obj + ".log"):
        with open(obj + ".log") as fh:
            log = fh.read()
    return obj, log


def build(verbose: bool = False) -> str:
    """Compile every csrc/*.cu for sm_103a and link libmla.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    hdr = _headers_digest()
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s, hdr, verbose), srcs))
    objs = [o for o, _ in results]
    if verbose:
        for o, log in results:
            if log:
                sys.stdout.write(f"== {os.path.basename(o)}\n{log}")
    link_key = hashlib.sha256("".join(objs).encode()).hexdigest()[:16]
    stamp = LIB + ".stamp"
    if os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == link_key:
        return LIB
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", LIB + ".tmp", *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link of libmla.so failed:\n{p.stdout}{p.stderr}")
    os.replace(LIB + ".tmp", LIB)
    with open(stamp, "w") as fh:
        fh.write(link_key)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
