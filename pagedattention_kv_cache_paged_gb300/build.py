"""Build libpagedattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Each translation unit under csrc/ compiles in parallel into _build/, then one link step writes
``pagedattention_kv_cache_paged_gb300/libpagedattn.so``.  Run ``python -m
pagedattention_kv_cache_paged_gb300.build`` or call :func:`build`.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libpagedattn.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedattn.so")


def sources() -> list:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if p.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + p.stdout)
    return p.stdout


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    """Compile stale translation units and link the library.  PAGEDATTN_NVCC_FLAGS (environment)
    adds compiler flags, e.g. -D overrides of kernel tuning constants; a change of flags rebuilds
    everything."""
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    user_flags = os.environ.get("PAGEDATTN_NVCC_FLAGS", "").split()
    stamp = os.path.join(BUILD_DIR, "flags.txt")
    old = open(stamp).read() if os.path.exists(stamp) else None
    if old != " ".join(user_flags):
        force = True
        with open(stamp, "w") as f:
            f.write(" ".join(user_flags))
    srcs = sources()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "pagedattn.h"))
    newest_header = max(os.path.getmtime(h) for h in headers)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    objs = []
    for src in srcs:
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        stale = (force or ptxas_info or not os.path.exists(obj)
                 or os.path.getmtime(obj) < max(os.path.getmtime(src), newest_header))
        if stale:
            jobs.append([nvcc, *ARCH, *CFLAGS, *user_flags, *extra, "-c", src, "-o", obj])
    outputs = []
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            outputs = list(ex.map(_run, jobs))
    if verbose or ptxas_info:
        for o in outputs:
            sys.stdout.write(o)
    if jobs or not os.path.exists(LIB_PATH):
        _run([nvcc, *ARCH, "-shared", "-o", LIB_PATH, *objs])
    return LIB_PATH


if __name__ == "__main__":
    path = build(verbose=True, ptxas_info="--ptxas" in sys.argv, force="--force" in sys.argv)
    print(path)
