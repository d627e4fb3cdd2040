"""Build libdspark.so for sm_103a with nvcc (in-tree, no torch extension).

Each translation unit is compiled in parallel, then linked into one shared
library under ``speculative_decoding_drafting_gb300/_build``.  A unit is
rebuilt only when it, a header, or the flags changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libdspark.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdspark.so")


def _digest(paths, extra: str) -> str:
    h = hashlib.sha256(extra.encode())
    for p in sorted(paths):
        with open(p, "rb") as f:
            h.update(p.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                     glob.glob(os.path.join(ROOT, "include", "*.h")))
    exe = nvcc()
    flag_key = " ".join([exe] + ARCH + FLAGS)
    hdr_digest = _digest(headers, flag_key)
    stamp = os.path.join(BUILD, "libdspark.stamp")
    full = _digest(sources + headers, flag_key)
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == full:
                return LIB

    def compile_one(src: str) -> str:
        name = os.path.splitext(os.path.basename(src))[0]
        obj = os.path.join(BUILD, f"{name}.{_digest([src], hdr_digest)}.o")
        if force or not os.path.exists(obj):
            tmp = obj + f".tmp{os.getpid()}"
            cmd = [exe] + ARCH + FLAGS + ["-c", src, "-o", tmp]
            if verbose:
                print(" ".join(cmd))
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, obj)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(sources), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [exe] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(full)
    # drop stale objects
    keep = set(objs)
    for o in glob.glob(os.path.join(BUILD, "*.o")):
        if o not in keep:
            try:
                os.remove(o)
            except OSError:
                pass
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
