"""Build libspectree.so in-tree with nvcc for sm_103a (GB300).

Every translation unit is compiled in parallel with one ``-gencode`` and linked into one shared
library next to this file.  No cmake, no setuptools: plain nvcc, so the same step runs on the x86
build host (cross-compiling) and on the aarch64 GPU host.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libspectree.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["spectree_abi.cu", "tree_attention.cu", "tree_verify.cu", "verify_noalloc.cu",
           "kv_compact.cu", "filter.cu", "tree_build.cu", "lm_head.cu", "verify_greedy.cu",
           "verify_head.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspectree")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra]


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs.append(os.path.join(ROOT, "include", "spectree.h"))
    return hdrs


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    hdrs = _deps()
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or not _newer(o, [s, *hdrs]):
            jobs.append([exe, *_flags(extra_flags), "-c", s, "-o", o])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        return r

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    if jobs or not _newer(LIB, objs):
        tmp = LIB + ".tmp"
        # cudart is linked statically; the driver API (tensor-map encoding) is reached through
        # cudaGetDriverEntryPoint, so the library does not link libcuda directly.
        run([exe, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
