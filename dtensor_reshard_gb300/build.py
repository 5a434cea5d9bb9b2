"""Build libreshard.so in-tree with nvcc for sm_103a (GB300).

The two translation units (host planner, CUDA kernels) compile in parallel and
link into ``dtensor_reshard_gb300/libreshard.so``; the CUDA runtime is linked
statically, so the library needs only the driver at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libreshard.so")
BUILD_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["planner.cpp", "batch.cpp", "kernels.cu", "bulk_fanout.cu", "transpose.cu",
           "static_scratch.cu", "realign_staged.cu", "refit.cpp", "partition.cpp"]
HEADERS = ["internal.h", "staging.cuh"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libreshard.so cannot be built")


def compile_flags(extra=()):
    return ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O3,-Wall",
            "-I" + INCLUDE, "-I" + CSRC, *extra]


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    """Compile and link libreshard.so; returns its path.  Raises on failure."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "reshard.h")]
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(d) for d in deps)):
        return LIB_PATH
    exe = nvcc()
    procs, objs = [], []
    for src in srcs:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        extra = ["-Xptxas", "-v"] if (ptxas_info and src.endswith(".cu")) else []
        cmd = [exe, *compile_flags(extra), "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
        objs.append(obj)
    logs = []
    for cmd, p in procs:
        out, _ = p.communicate()
        logs.append(out)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed ({p.returncode}): {' '.join(cmd)}\n{out}")
    tmp = LIB_PATH + ".tmp"
    link = [exe, "-shared", *ARCH, "-o", tmp, *objs]
    if verbose:
        print(" ".join(link), file=sys.stderr)
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose or ptxas_info:
        for out in logs:
            if out.strip():
                print(out, file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    build(verbose=True, ptxas_info="--ptxas" in sys.argv, force="--force" in sys.argv)
    print(LIB_PATH)
