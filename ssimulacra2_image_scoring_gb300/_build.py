"""Builds libss2.so in-tree with nvcc for sm_103a.

The translation units under ``csrc/`` are compiled in parallel into
``_build/`` and linked (static CUDA runtime) into ``_lib/libss2.so``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
SO_PATH = os.path.join(LIBDIR, "libss2.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libss2")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    if _stale(obj, [src, *headers(), __file__]):
        tmp = obj + f".tmp{os.getpid()}"
        subprocess.run([nvcc(), *NVFLAGS, *extra, "-c", src, "-o", tmp], check=True)
        os.replace(tmp, obj)
    return obj


def build(force: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compiles and links libss2.so; returns its path."""
    extra = list(extra_flags or [])
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            os.remove(os.path.join(BUILD, f))
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), srcs))
    if force or _stale(SO_PATH, objs):
        tmp = SO_PATH + f".tmp{os.getpid()}"
        subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "static", "-Xlinker",
                        "--no-undefined", "-o", tmp, *objs], check=True)
        os.replace(tmp, SO_PATH)
    return SO_PATH


if __name__ == "__main__":
    print(build())
