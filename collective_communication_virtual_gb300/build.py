"""Build libvcomm.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process, in parallel, then one nvcc
call links the shared library (CUDA runtime linked statically, so loading the library
needs no GPU).  A rebuild happens only when a source or header is newer than the
library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libvcomm.so")

SOURCES = ["vcomm.cpp", "planner.cpp", "ring_launch.cu", "k_onepass.cu", "k_onepass_small.cu", "k_group.cu", "k_tree.cu", "k_tree_more.cu",
           "k_copy.cu", "k_ring_simple.cu", "k_ring_ll.cu", "k_ring_ll128.cu", "noalloc.cu", "k_tma.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")


def _flags():
    return ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-Wall", *ARCH,
            f"-I{INCLUDE}", f"-I{CSRC}"]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "vcomm.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, "obj", src + ".o")
    cmd = [NVCC, *_flags(), "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas and src.endswith(".cu"):
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, jobs: int | None = None, verbose_ptxas: bool = False) -> str:
    """Compile every translation unit and link ``_build/libvcomm.so``; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(os.path.join(BUILD, "obj"), exist_ok=True)
    jobs = jobs or min(len(SOURCES), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([NVCC, "-shared", *ARCH, "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
